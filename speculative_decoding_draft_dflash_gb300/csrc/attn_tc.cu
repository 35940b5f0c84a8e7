// Block attention on tcgen05 tensor cores (bf16 path; bf16 or E4M3 cache).
//
// The R = G * bs block queries that share one KV head (G query heads x bs
// block positions, at most 128) form the rows of one M=128 MMA tile, so every
// cached K/V row read from HBM serves all of them (DFlash KV Injection
// Walkthrough, Step 4.4: non-causal, every block query sees every key;
// DFlash source guide (II), part 1: query head h reads KV head h / G).
//
// Three kernels:
//   attn_schedule_kernel   one CTA: from the cache lengths, lays the key ranges
//                          of all (sequence, KV head) pairs end to end as one
//                          stream of 128-key tiles, each range led by a cost
//                          for its item, and gives every SM an equal share of
//                          that cost, a range cut where a share ends;
//   attn_tc_kernel         persistent, one CTA per SM, each working through
//                          the items of its share in order. A split range
//                          leaves its output normalised in bf16 with its
//                          (max, sum);
//   attn_combine_kernel    merges the partial results of split ranges.
//
// attn_tc_kernel roles (warp: job):
//   0-3, 4-7   softmax. Warp w serves TMEM lanes 32(w%4)..+31 (query rows)
//              and S columns 64(w/4)..+63: two threads per row, exchanging the
//              tile maximum and the row sum through shared memory. P (bf16) is
//              stored into TMEM and read from there by the PV MMA.
//   8 (6)      TMA: the Q tile of each item (double-buffered) and K tiles
//              (three stages for R <= 64);
//   9 (7)      MMA: S_j = Q K_j^T (two TMEM S buffers), O += P_j V_j (P from
//              TMEM, V read MN-major from shared memory); S_{j+2} is issued
//              before PV_j;
//   10 (8)     TMA: V tiles (released later than K, so on their own thread;
//              the first waits for the first K tile, which the first S needs);
//   2,3,10,11  fp8 cache with R <= 64 only: V tile conversion to f16 (a twelfth
//              warp; the softmax leaves lane quarters 2-3 and their warps free).
// In parentheses: the warp with R <= 64 (for the V loads: fp8 cache with R <= 64),
// which keeps the single-thread roles off the two sub-partitions the softmax then
// runs on.
// O is rescaled in TMEM only when a row's running maximum grows by more than
// 2^8, so almost every tile skips it.
//
// fp8 (E4M3) cache (KV Cache + Speculative Decoding Interview Cheat Sheet,
// sections 2.1 and 4.5: one byte per cached element): the MMAs run as
// kind::f8f6f4 on the cached codes directly, so a tile is half the bytes of a
// bf16 one. Q and P carry about bf16 precision as two E4M3 terms each, the
// codes and the codes of the remainder (x ~ hi + lo), so S = Q_hi K^T + Q_lo K^T
// and O += P_hi V + P_lo V: twice the MMAs of half the width, the same tensor
// time as bf16. P is formed as 64 p with p <= 4 (rescale threshold 2^2), which
// keeps it inside E4M3's range and its small values normal. With R <= 64 the
// warps of lane quarters 2-3 convert V to f16 instead and PV runs as kind::f16
// with P in f16. The K scale folds into the score scale and the V scale into
// the output.
#include <float.h>

#include <mutex>

#include "attn_sched.cuh"
#include "sm100_ptx.cuh"

namespace dflash {
namespace {

constexpr int TK = 128;                    // keys per tile
constexpr uint32_t TILE = 128 * 128 * 2;   // 32 KB: one bf16 K or V tile (128 keys x 128 dims)
constexpr uint32_t HALF = TILE / 2;        // one 64-column swizzled box
constexpr int kSoftmaxWarps = 8;

constexpr uint32_t TM_S = 0, TM_O = 256, TM_P = 384;  // TMEM columns: S[2], O, P[2] (64 each)
constexpr int kRing = 4;                   // item ring slots

// Shared-memory plan. bf16, NARROW (R <= 64): query rows 64-127 of an A tile are
// padding, so the two Q buffers interleave (each only needs its rows 0-63 to be its
// own) and K gets a third stage: a K tile must land before its S MMA, which runs two
// tiles ahead of the PV MMA, so K loads need the longer lead. bf16, WIDE (R > 64):
// plain double buffers.
// fp8 (E4M3 cache): K / V tiles are 16 KB (one 128-byte row per key), so there is
// room for four K and three V stages. A Q buffer holds the code rows of Q, then the
// remainder-code rows (R rows of 128 B each, padded to 64 or 128); the S MMA reads
// 128 rows from either, and a NARROW buffer's rows 64-127 fall on what follows it
// (an 8 KB pad after the last one).
template <bool NARROW, bool FP8>
struct Plan {
  // fp8 with R <= 64: the warps of TMEM lane quarters 2 and 3 hold no query rows, so
  // they convert each V tile to f16 (zeroing rows past the key range) and the PV MMA
  // runs as kind::f16 with P in f16: one pack per two values instead of a code split.
  static constexpr bool CONV = FP8 && NARROW;
  // Warp roles. A warp issues on sub-partition (warp % 4), and only the warps of
  // sub-partition q can touch TMEM lanes 32q..32q+31. With R <= 64 the softmax lives on
  // sub-partitions 0-1, and the K/Q producer and the MMA issuer move to warps 6 and 7
  // (sub-partitions 2-3) instead of competing with the softmax for issue slots. bf16:
  // warps 2, 3, 8, 9 stay idle. fp8: four warps on sub-partitions 2-3 convert V (one key
  // row per thread), 2, 3 and a twelfth pair 10, 11, and the V producer moves to warp 8.
  static constexpr int W_KQ = NARROW ? 6 : 8, W_MMA = NARROW ? 7 : 9;
  static constexpr int W_V = CONV ? 8 : 10;
  // CONV: the V converters are warps 2, 3, 10 and 11 (a twelfth warp), so that the K/Q
  // producer and the MMA issuer keep sub-partitions 2-3 as with a bf16 cache
  static constexpr int THREADS = 32 * (kSoftmaxWarps + (CONV ? 4 : 3));
  static constexpr uint32_t TILE_B = FP8 ? TK * 128 : TILE;  // one K or V tile (as loaded)
  static constexpr int K_STAGES = FP8 ? 4 : (NARROW ? 3 : 2);
  static constexpr int V_STAGES = FP8 ? 3 : 2;
  static constexpr int C_STAGES = CONV ? 2 : 0;              // converted (f16) V tiles
  static constexpr int C_RING = CONV ? C_STAGES : 1;         // its ring size in index math
  static constexpr uint32_t QPART = NARROW ? 8192 : 16384;   // fp8: code rows of one buffer
  static constexpr uint32_t Q_BYTES = FP8 ? (NARROW ? 4 * QPART + 8192 : 4 * QPART)
                                          : (NARROW ? 40960 : 2 * TILE);
  static constexpr uint32_t Q_TX = FP8 ? 2 * QPART : (NARROW ? TILE / 2 : TILE);  // per Q load
  static constexpr uint32_t OFF_K = Q_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + K_STAGES * TILE_B;
  static constexpr uint32_t OFF_C = OFF_V + V_STAGES * TILE_B;
  static constexpr uint32_t OFF_BAR = OFF_C + C_STAGES * TILE;
  // mbarrier slots
  static constexpr int B_QF = 0, B_QE = 2, B_KF = 4, B_KE = B_KF + K_STAGES;
  static constexpr int B_VF = B_KE + K_STAGES, B_VE = B_VF + V_STAGES;
  static constexpr int B_CF = B_VE + V_STAGES, B_CE = B_CF + C_STAGES;
  static constexpr int B_SF = B_CE + C_STAGES, B_SE = B_SF + 2, B_P = B_SE + 2, B_PV = B_P + 2;
  static constexpr int B_ITF = B_PV + 2, B_ITE = B_ITF + kRing, B_FIN = B_ITE + kRing;
  static constexpr int N_BARS = B_FIN + 1;
  static constexpr uint32_t OFF_RING = OFF_BAR + ((8 * N_BARS + 15) & ~15);
  static constexpr size_t SMEM = 1024 + OFF_RING + 16 * kRing;
  // O is rescaled only when a row's running maximum grows by more than 2^this. fp8 with
  // P in E4M3 codes: P is stored as 64 p, and p <= 4 keeps 64 p inside E4M3's range (448).
  static constexpr bool P_CODES = FP8 && !CONV;
  static constexpr float RESCALE_LOG2 = P_CODES ? 2.0f : 8.0f;
  __device__ static uint32_t q_base(int buf) {
    return FP8 ? buf * 2 * QPART : (NARROW ? buf * 8192u : buf * TILE);
  }
};

struct AttnTcParams {
  CUtensorMap q;   // [B*n_h*bs][128] bf16, box rows 64 (NARROW) or 128; fp8: the Q codes
  CUtensorMap q_lo;  // fp8: the Q remainder codes (same shape)
  CUtensorMap k;   // [B*n_kv*capacity][128] bf16 or E4M3 (this layer)
  CUtensorMap v;
  const int32_t* table;   // paged cache: [batch][pps] page ids of 128-row pages, or null
  int pps;
  const int32_t* qstart;  // [batch]: first position of each block (window test)
  int32_t* lens;          // [batch]: receives lens_new once the attention is done
  const int32_t* lens_new;
  bf16* out;
  float* part_acc;       // [pair][max_splits][R][128] bf16: a split's normalised output
  float2* part_ml;       // [pair][max_splits][R]
  const int4* items;     // [grid] first item of each CTA (the last of its share), then
                         // the list: {pair, k_begin, k_end, split (-1 = whole range)}
  const int* first;      // [grid + 1]: CTA c takes list items first[c] .. first[c + 1] - 1
  unsigned* status;
  int batch, n_h, n_kv, bs, G, R, capacity, window, table_len, max_splits;
  float sl2;      // scaling * log2(e) (fp8: times k_scale)
  float v_scale;  // fp8: scale of the V codes
  int out_v8;     // out is 32-byte aligned: rows leave in 32-byte stores
  unsigned long long wait_ns;  // limit of the pipeline waits (2 s unless a test lowers it)
  int* list_ready;  // the work list's "complete" flag: cleared for the next list
};

__device__ __forceinline__ void drain(uint32_t bar, uint32_t parity, unsigned* status) {
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer() - t0 > ptx::kWaitLimitNs) {
      atomicOr(status, DFLASH_DEV_TIMEOUT);
      return;
    }
  }
}

// First row of the 128-key tile starting at key k0 (a multiple of 128 when paged) of
// (sequence b, KV head kvh) in the K / V tensor maps.
__device__ __forceinline__ int tile_row(const AttnTcParams& p, int b, int kvh, int k0) {
  if (p.table) return (p.table[b * p.pps + (k0 >> 7)] * p.n_kv + kvh) * TK;
  return (b * p.n_kv + kvh) * p.capacity + k0;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// TS form: A from tensor memory, B from a shared-memory descriptor.
__device__ __forceinline__ void mma_bf16_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// kind::f8f6f4 (E4M3 x E4M3, fp32 accumulator, K = 32 per instruction): SS and TS forms.
__device__ __forceinline__ void mma_f8(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_f8_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor: kind::f16 with A = B = f16, D = f32, both K-major, M x N.
constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ uint32_t pack_f16(float a, float b) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));  // a -> low half
  return r;
}

// Two E4M3 codes (low byte first) -> f16x2 (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((uint16_t)two));
  return r;
}

// Instruction descriptor: kind::f8f6f4, A = B = E4M3, D = f32, both K-major, M x N.
constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// 32 lanes x 16 columns of 32-bit TMEM cells.
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

// ---------------------------------------------------------------------------
// work list: one CTA (attn_sched.cuh), unless the projection launch built it
// ---------------------------------------------------------------------------
static_assert(TK == sched::kTileKeys, "attention tile and work-list tile differ");

__global__ void __launch_bounds__(1024) attn_schedule_kernel(sched::Params p) { sched::build(p); }

// ---------------------------------------------------------------------------
// attention
// ---------------------------------------------------------------------------
template <bool NARROW, bool FP8>
__global__ void __launch_bounds__(Plan<NARROW, FP8>::THREADS, 1) attn_tc_kernel(const __grid_constant__ AttnTcParams p) {
  using PL = Plan<NARROW, FP8>;
  constexpr int NCOL = 64;  // S columns per softmax thread
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(smem + PL::OFF_BAR);
  int4* ring = (int4*)(smem + PL::OFF_RING);
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ float xch[2][2][128];  // tile maxima of the two column halves
  __shared__ float xl[2][128];      // row sums of the two column halves

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nq = (p.R + 31) >> 5;                 // TMEM lane quarters holding query rows
  const int n_soft = 64 * nq;                     // softmax threads
  const bool soft = warp < kSoftmaxWarps && (warp & 3) < nq;
  // V converters (PL::CONV): the warps of lane quarters 2 and 3, one key row per thread
  const bool conv = PL::CONV && (warp & 3) >= 2 && (warp < 4 || warp >= 10);
  constexpr int kConv = PL::CONV ? 128 : 0;
  const uint32_t sbase = ptx::smem_u32(smem);
  // barriers (8 bytes each): q 2+2, k and v full+empty per stage, s 2+2, p 2, pv 2,
  // items 4+4, MMA exit 1
  const uint32_t q_full0 = ptx::smem_u32(bars + PL::B_QF), q_empty0 = ptx::smem_u32(bars + PL::B_QE);
  const uint32_t k_full0 = ptx::smem_u32(bars + PL::B_KF), k_empty0 = ptx::smem_u32(bars + PL::B_KE);
  const uint32_t v_full0 = ptx::smem_u32(bars + PL::B_VF), v_empty0 = ptx::smem_u32(bars + PL::B_VE);
  const uint32_t c_full0 = ptx::smem_u32(bars + PL::B_CF), c_empty0 = ptx::smem_u32(bars + PL::B_CE);
  const uint32_t s_full0 = ptx::smem_u32(bars + PL::B_SF), s_free0 = ptx::smem_u32(bars + PL::B_SE);
  const uint32_t p_full0 = ptx::smem_u32(bars + PL::B_P), pv_done0 = ptx::smem_u32(bars + PL::B_PV);
  const uint32_t it_full0 = ptx::smem_u32(bars + PL::B_ITF), it_empty0 = ptx::smem_u32(bars + PL::B_ITE);
  const uint32_t mma_fin = ptx::smem_u32(bars + PL::B_FIN);

  if (threadIdx.x == 0) {
    // the projection launch that may have prefetched from the list has finished
    if (blockIdx.x == 0 && p.list_ready) *p.list_ready = 0;
    abort_flag = 0;
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(q_full0 + 8 * i, 1);
      ptx::mbar_init(q_empty0 + 8 * i, 1);
      ptx::mbar_init(s_full0 + 8 * i, 1);
      ptx::mbar_init(s_free0 + 8 * i, n_soft);
      ptx::mbar_init(pv_done0 + 8 * i, 1);
    }
    for (int i = 0; i < PL::K_STAGES; ++i) {
      ptx::mbar_init(k_full0 + 8 * i, 1);
      ptx::mbar_init(k_empty0 + 8 * i, 1);
    }
    for (int i = 0; i < PL::V_STAGES; ++i) {
      ptx::mbar_init(v_full0 + 8 * i, 1);
      ptx::mbar_init(v_empty0 + 8 * i, PL::CONV ? kConv : 1);  // converters read the tile
    }
    for (int i = 0; i < PL::C_STAGES; ++i) {
      ptx::mbar_init(c_full0 + 8 * i, kConv);
      ptx::mbar_init(c_empty0 + 8 * i, 1);
    }
    // one per P buffer: the softmax may finish tiles g and g + 1 before the MMA thread
    // looks for tile g, but not tile g + 2 (that needs PV_g)
    ptx::mbar_init(p_full0, n_soft);
    ptx::mbar_init(p_full0 + 8, n_soft);
    ptx::mbar_init(mma_fin, 1);
    for (int i = 0; i < kRing; ++i) {
      ptx::mbar_init(it_full0 + 8 * i, 1);
      ptx::mbar_init(it_empty0 + 8 * i, 2 + n_soft + kConv);
    }
    ptx::fence_mbar_init();
  }
  if (warp == PL::W_MMA) {
    ptx::tmem_alloc(ptx::smem_u32(&tmem_slot), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == PL::W_KQ) {
    // ---------------------------------------------------- item fetch, Q and K loads
    if (lane == 0) {
      ptx::prefetch_tmap(&p.q);
      if (FP8) ptx::prefetch_tmap(&p.q_lo);
      ptx::prefetch_tmap(&p.k);
      ptx::prefetch_tmap(&p.v);
      const uint64_t pol = ptx::policy_evict_first();
      int gk = 0, n = 0, nq_loads = 0;
      // this CTA's items f0 .. f1 - 1 of the list, the last one first (the two ends of a
      // share are the ranges cut at its boundaries; taking both early leaves the whole
      // ranges, which need no merge, for the end). The first item has a slot of its own,
      // so that reading it does not wait for the list bounds; the others are read one
      // item ahead.
      const int4* list = p.items + gridDim.x;
      const int f0 = p.first[blockIdx.x], f1 = p.first[blockIdx.x + 1];
      int4 it_next = p.items[blockIdx.x];
      bool stop = false;
      for (;; ++n) {
        const int slot = n % kRing;
        if (n >= kRing &&
            !ptx::mbar_wait(it_empty0 + 8 * slot, ((n / kRing) - 1) & 1, &abort_flag, p.status, p.wait_ns))
          break;
        const int4 it = it_next;
        ring[slot] = it;
        ptx::mbar_arrive(it_full0 + 8 * slot);  // release: the ring entry is visible to waiters
        if (it.x < 0) break;
        it_next = f0 + n + 1 < f1 ? list[f0 + n] : make_int4(-1, 0, 0, 0);
        const int b = it.x / p.n_kv, kvh = it.x - b * p.n_kv;
        const int qb = n & 1;
        if (n >= 2 && !ptx::mbar_wait(q_empty0 + 8 * qb, ((n >> 1) - 1) & 1, &abort_flag, p.status, p.wait_ns))
          break;
        const int qrow = (b * p.n_h + kvh * p.G) * p.bs;
        const uint32_t qd = sbase + PL::q_base(qb);
        ptx::mbar_arrive_expect_tx(q_full0 + 8 * qb, PL::Q_TX);
        ptx::tma_load_2d(qd, &p.q, q_full0 + 8 * qb, 0, qrow);
        if (FP8)
          ptx::tma_load_2d(qd + PL::QPART, &p.q_lo, q_full0 + 8 * qb, 0, qrow);
        else
          ptx::tma_load_2d(qd + HALF, &p.q, q_full0 + 8 * qb, 64, qrow);
        ++nq_loads;
        const int ntiles = (it.z - it.y + TK - 1) / TK;
        int row_next = tile_row(p, b, kvh, it.y);  // the next tile's row, fetched a tile ahead
        for (int j = 0; j < ntiles; ++j) {
          const int row = row_next;
          if (j + 1 < ntiles) row_next = tile_row(p, b, kvh, it.y + (j + 1) * TK);
          const int s = gk % PL::K_STAGES, u = gk / PL::K_STAGES;
          if (gk >= PL::K_STAGES &&
              !ptx::mbar_wait(k_empty0 + 8 * s, (u - 1) & 1, &abort_flag, p.status, p.wait_ns)) {
            stop = true;
            break;
          }
          const uint32_t kd = sbase + PL::OFF_K + s * PL::TILE_B;
          ptx::mbar_arrive_expect_tx(k_full0 + 8 * s, PL::TILE_B);
          ptx::tma_load_2d_hint(kd, &p.k, k_full0 + 8 * s, 0, row, pol);
          if (!FP8) ptx::tma_load_2d_hint(kd + HALF, &p.k, k_full0 + 8 * s, 64, row, pol);
          ++gk;
        }
        if (stop) break;
      }
      // nothing of ours may still be landing in shared memory when the CTA exits
      for (int i = nq_loads > 2 ? nq_loads - 2 : 0; i < nq_loads; ++i)
        drain(q_full0 + 8 * (i & 1), (i >> 1) & 1, p.status);
      for (int g = gk > PL::K_STAGES ? gk - PL::K_STAGES : 0; g < gk; ++g)
        drain(k_full0 + 8 * (g % PL::K_STAGES), (g / PL::K_STAGES) & 1, p.status);
    }
  } else if (warp == PL::W_V) {
    // ---------------------------------------------------- V loads
    if (lane == 0) {
      const uint64_t pol = ptx::policy_evict_first();
      int gv = 0;
      bool stop = false;
      for (int n = 0; !stop; ++n) {
        const int slot = n % kRing;
        if (!ptx::mbar_wait(it_full0 + 8 * slot, (n / kRing) & 1, &abort_flag, p.status, p.wait_ns)) break;
        const int4 it = ring[slot];
        ptx::mbar_arrive(it_empty0 + 8 * slot);
        if (it.x < 0) break;
        // At the start every CTA asks HBM for its first tiles at once, and the first S
        // needs only Q and K_0: V waits until K_0 has landed, so that it is not queued
        // ahead of it (V_0 is needed only after the first tile's softmax).
        if (n == 0 && !ptx::mbar_wait(k_full0, 0, &abort_flag, p.status, p.wait_ns)) break;
        const int b = it.x / p.n_kv, kvh = it.x - b * p.n_kv;
        const int ntiles = (it.z - it.y + TK - 1) / TK;
        int row_next = tile_row(p, b, kvh, it.y);
        for (int j = 0; j < ntiles; ++j) {
          const int row = row_next;
          if (j + 1 < ntiles) row_next = tile_row(p, b, kvh, it.y + (j + 1) * TK);
          const int s = gv % PL::V_STAGES, u = gv / PL::V_STAGES;
          if (gv >= PL::V_STAGES &&
              !ptx::mbar_wait(v_empty0 + 8 * s, (u - 1) & 1, &abort_flag, p.status, p.wait_ns)) {
            stop = true;
            break;
          }
          const uint32_t vd = sbase + PL::OFF_V + s * PL::TILE_B;
          ptx::mbar_arrive_expect_tx(v_full0 + 8 * s, PL::TILE_B);
          ptx::tma_load_2d_hint(vd, &p.v, v_full0 + 8 * s, 0, row, pol);
          if (!FP8) ptx::tma_load_2d_hint(vd + HALF, &p.v, v_full0 + 8 * s, 64, row, pol);
          ++gv;
        }
      }
      for (int g = gv > PL::V_STAGES ? gv - PL::V_STAGES : 0; g < gv; ++g)
        drain(v_full0 + 8 * (g % PL::V_STAGES), (g / PL::V_STAGES) & 1, p.status);
    }
  } else if (warp == PL::W_MMA) {
    // ---------------------------------------------------- MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc_s = FP8 ? idesc_e4m3_f32(128, TK) : ptx::idesc_bf16_f32(128, TK);
      constexpr uint32_t idesc_pv =  // V MN-major
          (PL::P_CODES ? idesc_e4m3_f32(128, 128)
                       : PL::CONV ? idesc_f16_f32(128, 128) : ptx::idesc_bf16_f32(128, 128)) |
          (1u << 16);
      int gt = 0;
      bool stop = false, issued = false;
      for (int n = 0; !stop; ++n) {
        const int slot = n % kRing;
        if (!ptx::mbar_wait(it_full0 + 8 * slot, (n / kRing) & 1, &abort_flag, p.status, p.wait_ns)) break;
        const int4 it = ring[slot];
        ptx::mbar_arrive(it_empty0 + 8 * slot);
        if (it.x < 0) break;
        const int qb = n & 1;
        if (!ptx::mbar_wait(q_full0 + 8 * qb, (n >> 1) & 1, &abort_flag, p.status, p.wait_ns)) break;
        const int T = (it.z - it.y + TK - 1) / TK, base = gt;
        const uint32_t qa = sbase + PL::q_base(qb);
        auto issue_s = [&](int j) -> bool {
          const int g = base + j, s = g & 1, u = g >> 1;
          const int ks = g % PL::K_STAGES, ku = g / PL::K_STAGES;
          if (g >= 2 && !ptx::mbar_wait(s_free0 + 8 * s, (u - 1) & 1, &abort_flag, p.status, p.wait_ns))
            return false;
          if (!ptx::mbar_wait(k_full0 + 8 * ks, ku & 1, &abort_flag, p.status, p.wait_ns)) return false;
          ptx::tc_fence_after();
          const uint32_t ka = sbase + PL::OFF_K + ks * PL::TILE_B;
          if (FP8) {
            // S = Qcodes K^T + Qremainder K^T: 4 K-steps of 32 dims each
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_f8(tmem + TM_S + s * TK,
                     ptx::smem_desc_sw128(qa + (kk >> 2) * PL::QPART + (kk & 3) * 32),
                     ptx::smem_desc_sw128(ka + (kk & 3) * 32), idesc_s, kk > 0 ? 1u : 0u);
          } else {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t off = (kk >> 2) * HALF + (kk & 3) * 32;
              ptx::mma_bf16(tmem + TM_S + s * TK, ptx::smem_desc_sw128(qa + off),
                            ptx::smem_desc_sw128(ka + off), idesc_s, kk > 0 ? 1u : 0u);
            }
          }
          issued = true;
          ptx::mma_commit(k_empty0 + 8 * ks);
          ptx::mma_commit(s_full0 + 8 * s);
          if (j == T - 1) ptx::mma_commit(q_empty0 + 8 * qb);
          return true;
        };
        if (!issue_s(0) || (T > 1 && !issue_s(1))) break;
        for (int j = 0; j < T; ++j) {
          // S of tile j + 2 goes first: its buffer is free once the softmax has read S_j
          // (early in that tile's softmax), while PV_j waits for the end of it; issued the
          // other way round, each S would queue behind a PV that waited for a softmax.
          if (j + 2 < T && !issue_s(j + 2)) {
            stop = true;
            break;
          }
          const int g = base + j;
          // the V tile: as loaded, or (CONV) its f16 conversion
          const int vs = PL::CONV ? g % PL::C_STAGES : g % PL::V_STAGES;
          const int vu = PL::CONV ? g / PL::C_STAGES : g / PL::V_STAGES;
          const uint32_t vfull = PL::CONV ? c_full0 : v_full0;
          if (!ptx::mbar_wait(p_full0 + 8 * (g & 1), (g >> 1) & 1, &abort_flag, p.status, p.wait_ns) ||
              !ptx::mbar_wait(vfull + 8 * vs, vu & 1, &abort_flag, p.status, p.wait_ns)) {
            stop = true;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t va = PL::CONV ? sbase + PL::OFF_C + vs * TILE
                                       : sbase + PL::OFF_V + vs * PL::TILE_B;
          const uint32_t pa = tmem + TM_P + (g & 1) * 64;
          // Keys past the range end in the last tile (their P is 0): the MMA stops after the
          // last K-step that holds a key, and that step's rows past the end are zeroed
          // first (slots past the cache length may hold anything, and 0 * NaN would poison
          // O). The f16 conversion of a CONV tile already wrote those rows as zeros.
          constexpr int KS = PL::P_CODES ? 32 : 16;  // keys per K-step
          int key_end = TK;
          if (!PL::CONV && j == T - 1) {
            const int nvalid = it.z - (it.y + j * TK);
            if (nvalid < TK) {
              key_end = (nvalid + KS - 1) / KS * KS;
              uint4* vz = reinterpret_cast<uint4*>(smem + PL::OFF_V + vs * PL::TILE_B);
              for (int h = 0; h < (FP8 ? 1 : 2); ++h)  // bf16: two 64-column halves
                for (int c = nvalid * 8; c < key_end * 8; ++c) vz[h * (HALF / 16) + c] = make_uint4(0u, 0u, 0u, 0u);
              ptx::fence_proxy_async_smem();
            }
          }
          if (PL::P_CODES) {
            // O += Pcodes V + Premainder V: P columns 0-31 and 32-63, 32 keys per K-step
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              if ((kk & 3) * KS < key_end)
                mma_f8_ts(tmem + TM_O, pa + (kk >> 2) * 32 + (kk & 3) * 8,
                          ptx::smem_desc_sw128_mn(va + (kk & 3) * 4096, PL::TILE_B), idesc_pv,
                          (j > 0 || kk > 0) ? 1u : 0u);
          } else {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              if (kk * KS < key_end)
                mma_bf16_ts(tmem + TM_O, pa + kk * 8, ptx::smem_desc_sw128_mn(va + kk * 2048, HALF),
                            idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
          }
          ptx::mma_commit((PL::CONV ? c_empty0 : v_empty0) + 8 * vs);
          ptx::mma_commit(pv_done0 + 8 * (g & 1));
        }
        gt = base + T;
      }
      // every MMA issued by this thread (also those of an item cut short by an abort)
      // has finished before TMEM is released
      if (issued) {
        ptx::mma_commit(mma_fin);
        drain(mma_fin, 0, p.status);
      }
    }
  } else if (conv) {
    // ---------------------------------------------------- V conversion (E4M3 -> f16)
    // thread = key row k of the tile: 8 chunks of 16 codes -> 16 chunks of 8 f16 values,
    // both tiles in the 128-byte swizzled layout the MMA reads (chunk c of row k at
    // c ^ (k & 7)); rows past the key range are written as zeros
    const int k = (warp >= 10 ? 64 : 0) + ((warp & 3) - 2) * 32 + lane;
    const int sw = k & 7;
    int gv = 0;
    for (int n = 0;; ++n) {
      const int slot = n % kRing;
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(it_full0 + 8 * slot, (n / kRing) & 1, &abort_flag, p.status, p.wait_ns)))
        break;
      const int4 it = ring[slot];
      ptx::mbar_arrive(it_empty0 + 8 * slot);
      if (it.x < 0) break;
      const int T = (it.z - it.y + TK - 1) / TK;
      bool alive = true;
      for (int j = 0; j < T; ++j) {
        const int g = gv + j, vs = g % PL::V_STAGES, cs = g % PL::C_RING;
        alive = __all_sync(0xffffffffu, ptx::mbar_wait(v_full0 + 8 * vs, (g / PL::V_STAGES) & 1,
                                                       &abort_flag, p.status, p.wait_ns));
        if (alive && g >= PL::C_RING)
          alive = __all_sync(0xffffffffu, ptx::mbar_wait(c_empty0 + 8 * cs, ((g / PL::C_RING) - 1) & 1,
                                                         &abort_flag, p.status, p.wait_ns));
        if (!alive) break;
        const uint8_t* src = smem + PL::OFF_V + vs * PL::TILE_B + k * 128;
        uint8_t* dst = smem + PL::OFF_C + cs * TILE + k * 128;
        const bool valid = it.y + j * TK + k < it.z;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 x = valid ? *reinterpret_cast<const uint4*>(src + ((c ^ sw) << 4))
                                : make_uint4(0, 0, 0, 0);
          uint4 lo, hi;
          lo.x = e4m3x2_to_f16x2(x.x);
          lo.y = e4m3x2_to_f16x2(x.x >> 16);
          lo.z = e4m3x2_to_f16x2(x.y);
          lo.w = e4m3x2_to_f16x2(x.y >> 16);
          hi.x = e4m3x2_to_f16x2(x.z);
          hi.y = e4m3x2_to_f16x2(x.z >> 16);
          hi.z = e4m3x2_to_f16x2(x.w);
          hi.w = e4m3x2_to_f16x2(x.w >> 16);
          const int h = c >> 2, c2 = 2 * (c & 3);  // f16 half (64 dims) and its chunk
          *reinterpret_cast<uint4*>(dst + h * HALF + ((c2 ^ sw) << 4)) = lo;
          *reinterpret_cast<uint4*>(dst + h * HALF + (((c2 + 1) ^ sw) << 4)) = hi;
        }
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(c_full0 + 8 * cs);
        ptx::mbar_arrive(v_empty0 + 8 * vs);
      }
      if (!alive) break;
      gv += T;
    }
  } else if (soft) {
    // ---------------------------------------------------- softmax
    const int rt = (warp & 3) * 32 + lane;          // TMEM lane = query row g * bs + t
    const int half = warp >> 2;                      // S columns 64 * half .. + 63
    const int coff = half * NCOL;
    const bool rvalid = rt < p.R;
    const int gq = rvalid ? rt / p.bs : 0, t = rvalid ? rt - gq * p.bs : 0;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    int gt = 0;
    float s[NCOL];
    // Abort safety: the softmax threads meet at named barriers, which do not time out, so
    // a thread whose wait gave up never leaves on its own. It skips its work up to the next
    // barrier, whose OR of "gave up" flags then sends every softmax thread out together.
    for (int n = 0;; ++n) {
      const int slot = n % kRing;
      const bool got = __all_sync(0xffffffffu, ptx::mbar_wait(it_full0 + 8 * slot, (n / kRing) & 1, &abort_flag, p.status, p.wait_ns));
      if (ptx::named_sync_or(2, n_soft, !got)) break;
      const int4 it = ring[slot];
      ptx::mbar_arrive(it_empty0 + 8 * slot);
      if (it.x < 0) break;
      const int b = it.x / p.n_kv, kvh = it.x - b * p.n_kv;
      const int T = (it.z - it.y + TK - 1) / TK;
      const int qpos = p.qstart[b] + t;
      float m_ref = -INFINITY, l = 0.f;
      bool alive = true, dead = false;
      for (int j = 0; j < T; ++j) {
        const int g = gt + j, sb = g & 1, u = g >> 1;
        if (alive)
          alive = __all_sync(0xffffffffu, ptx::mbar_wait(s_full0 + 8 * sb, u & 1, &abort_flag, p.status, p.wait_ns));
        float mx = -INFINITY;
        if (alive) {
          ptx::tc_fence_after();
#pragma unroll
          for (int cc = 0; cc < NCOL / 32; ++cc) {
            uint32_t v[32];
            ptx::tmem_ld_32x32b_x32(tmem + lane_base + TM_S + sb * TK + coff + cc * 32, v);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) s[cc * 32 + e] = __uint_as_float(v[e]);
          }
          ptx::tc_fence_before();
          ptx::mbar_arrive(s_free0 + 8 * sb);
          // raw tile maximum over this thread's columns (masked keys -> -inf)
          const int key0 = it.y + j * TK + coff;
          const bool full = rvalid && key0 + NCOL <= it.z && (p.window <= 0 || qpos - key0 < p.window);
          if (full) {
            // three-input max: half the instructions of a pairwise chain (the softmax
            // sub-partitions are bound by instruction issue)
            float m4[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
            for (int e = 4; e < NCOL; e += 8) {
              m4[0] = fmax3(m4[0], s[e], s[e + 1]);
              m4[1] = fmax3(m4[1], s[e + 2], s[e + 3]);
              m4[2] = fmax3(m4[2], s[e + 4], s[e + 5]);
              m4[3] = fmax3(m4[3], s[e + 6], s[e + 7]);
            }
            mx = fmax3(m4[0], m4[1], fmaxf(m4[2], m4[3]));
          } else {
#pragma unroll
            for (int e = 0; e < NCOL; ++e) {
              const int key = key0 + e;
              const bool vis = rvalid && key < it.z && (p.window <= 0 || qpos - key < p.window);
              s[e] = vis ? s[e] : -INFINITY;
              mx = fmaxf(mx, s[e]);
            }
          }
        }
        xch[j & 1][half][rt] = mx;
        if (ptx::named_sync_or(2, n_soft, !alive)) {
          dead = true;
          break;
        }
        do {  // the rest of the tile; a wait that gives up leaves it (break) for the next barrier
        mx = fmaxf(mx, xch[j & 1][half ^ 1][rt]) * p.sl2;  // log2 domain
        float alpha = 1.f;
        bool resc = false;
        if (m_ref == -INFINITY) {
          m_ref = mx;                      // nothing accumulated yet for this row
        } else if (mx > m_ref + PL::RESCALE_LOG2) {
          alpha = ptx::ex2(m_ref - mx);
          m_ref = mx;
          resc = true;
        }
        // P in E4M3 codes: P = 64 p (2^6), whose small values stay normal E4M3 numbers
        const float mu = ((m_ref == -INFINITY) ? 0.f : m_ref) - (PL::P_CODES ? 6.f : 0.f);
        const float2 sl2v = make_float2(p.sl2, p.sl2), nmu = make_float2(-mu, -mu);
        float2 acc2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                          make_float2(0.f, 0.f)};
        uint32_t pk[NCOL / 2];
#pragma unroll
        for (int e = 0; e < NCOL; e += 2) {
          const float2 x = __ffma2_rn(make_float2(s[e], s[e + 1]), sl2v, nmu);
          const float2 y = make_float2(ptx::ex2(x.x), ptx::ex2(x.y));
          acc2[(e >> 1) & 3] = __fadd2_rn(acc2[(e >> 1) & 3], y);
          if (PL::P_CODES) {
            s[e] = y.x;
            s[e + 1] = y.y;
          } else {
            pk[e >> 1] = PL::CONV ? pack_f16(y.x, y.y) : pack_bf16(y.x, y.y);
          }
        }
        const float2 a01 = __fadd2_rn(acc2[0], acc2[1]), a23 = __fadd2_rn(acc2[2], acc2[3]);
        l = l * alpha + ((a01.x + a01.y) + (a23.x + a23.y));
        if (__any_sync(0xffffffffu, resc) && j > 0) {
          // O holds tiles < j once the previous PV is done; scale this thread's columns
          alive = __all_sync(0xffffffffu, ptx::mbar_wait(pv_done0 + 8 * ((g - 1) & 1), ((g - 1) >> 1) & 1, &abort_flag, p.status, p.wait_ns));
          if (!alive) break;
          ptx::tc_fence_after();
#pragma unroll 1
          for (int cc = 0; cc < NCOL / 32; ++cc) {
            uint32_t v[32];
            ptx::tmem_ld_32x32b_x32(tmem + lane_base + TM_O + coff + cc * 32, v);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
            ptx::tmem_st_32x32b_x32(tmem + lane_base + TM_O + coff + cc * 32, v);
          }
          ptx::tmem_st_wait();
        }
        // P buffer g & 1 is free once the PV of tile g - 2 is done
        if (g >= 2) {
          alive = __all_sync(0xffffffffu, ptx::mbar_wait(pv_done0 + 8 * sb, ((g - 2) >> 1) & 1, &abort_flag, p.status, p.wait_ns));
          if (!alive) break;
          ptx::tc_fence_after();
        }
        if (PL::P_CODES) {
          // codes of P (columns 0-31 of the buffer) and of its remainder (32-63)
          uint32_t hi[NCOL / 4], lo[NCOL / 4];
#pragma unroll
          for (int c = 0; c < NCOL / 4; ++c)
            e4m3x4_split(s[4 * c], s[4 * c + 1], s[4 * c + 2], s[4 * c + 3], hi[c], lo[c]);
          tmem_st_32x32b_x16(tmem + lane_base + TM_P + sb * 64 + half * 16, hi);
          tmem_st_32x32b_x16(tmem + lane_base + TM_P + sb * 64 + 32 + half * 16, lo);
        } else {
          ptx::tmem_st_32x32b_x32(tmem + lane_base + TM_P + sb * 64 + half * 32, pk);
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        ptx::mbar_arrive(p_full0 + 8 * sb);
        } while (false);
      }
      if (dead) break;
      gt += T;
      // ---- epilogue: this thread's 64 columns of O for this item
      xl[half][rt] = l;
      if (ptx::named_sync_or(2, n_soft, !alive)) break;
      l += xl[half ^ 1][rt];
      const int gl = gt - 1;
      // a wait that gives up here skips this item's stores; the next item's barrier ends it
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(pv_done0 + 8 * (gl & 1), (gl >> 1) & 1, &abort_flag, p.status, p.wait_ns)))
        continue;
      ptx::tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < NCOL / 32; ++cc) {
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(tmem + lane_base + TM_O + coff + cc * 32, v);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) s[cc * 32 + e] = __uint_as_float(v[e]);
      }
      ptx::tc_fence_before();
      if (!rvalid) continue;
      // this thread's 64 columns of the row, O / l in bf16: 32-byte stores (a full sector
      // each) when the destination allows, else 16-byte ones
      const float inv = l > 0.f ? (FP8 ? p.v_scale : 1.f) / l : 0.f;
      auto store_row = [&](bf16* dst, bool v8) {
        if (v8) {
#pragma unroll
          for (int k = 0; k < NCOL / 16; ++k) {
            uint32_t w[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) w[j] = pack_bf16(s[16 * k + 2 * j] * inv, s[16 * k + 2 * j + 1] * inv);
            ptx::st_global_v8(dst + 16 * k, w);
          }
        } else {
#pragma unroll
          for (int k = 0; k < NCOL / 8; ++k) {
            uint4 w;
            w.x = pack_bf16(s[8 * k + 0] * inv, s[8 * k + 1] * inv);
            w.y = pack_bf16(s[8 * k + 2] * inv, s[8 * k + 3] * inv);
            w.z = pack_bf16(s[8 * k + 4] * inv, s[8 * k + 5] * inv);
            w.w = pack_bf16(s[8 * k + 6] * inv, s[8 * k + 7] * inv);
            reinterpret_cast<uint4*>(dst)[k] = w;
          }
        }
      };
      if (it.w < 0) {
        store_row(p.out + ((size_t)(b * p.bs + t) * p.n_h + kvh * p.G + gq) * 128 + coff, p.out_v8 != 0);
      } else {
        // a split range's partial: its normalised output O / l (bf16, like the final rows)
        // and its (maximum, sum); the combine weights each by 2^(max - M) * sum (the
        // workspace is 256-byte aligned)
        const size_t prow = ((size_t)it.x * p.max_splits + it.w) * p.R + rt;
        store_row(reinterpret_cast<bf16*>(p.part_acc) + prow * 128 + coff, true);
        if (half == 0) p.part_ml[prow] = make_float2(m_ref, l);
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == PL::W_MMA) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// combine: one warp per (pair, query row)
// ---------------------------------------------------------------------------
// One query row of a marked pair: log-sum-exp merge of its split partials, or zeros
// for a refused sequence.
__device__ __forceinline__ void combine_row(const AttnTcParams& p, int n, int pr, int r, int lane) {
  const int b = pr / p.n_kv, kvh = pr - b * p.n_kv;
  const int gq = r / p.bs, t = r - gq * p.bs;
  bf16* orow = p.out + ((size_t)(b * p.bs + t) * p.n_h + kvh * p.G + gq) * 128;
  float o[4] = {0.f, 0.f, 0.f, 0.f};
  if (n > 1) {
    // each split holds its normalised output (bf16) and (max, sum): the row is
    // sum_c w_c out_c / sum_c w_c with w_c = 2^(max_c - M) sum_c. Lane c loads split c's
    // (max, sum) once (further splits in lane-strided passes) and hands its weight to the
    // others by shuffle; the rows of the first kPre splits are requested before all that.
    constexpr int kPre = 4;
    const size_t base = (size_t)pr * p.max_splits * p.R + r;
    const uint2* acc = reinterpret_cast<const uint2*>(reinterpret_cast<const bf16*>(p.part_acc) + base * 128) + lane;
    const size_t acc_stride = (size_t)p.R * 32;  // one split, in 4-value groups
    uint2 pre[kPre];
#pragma unroll
    for (int c = 0; c < kPre; ++c) pre[c] = c < n ? acc[c * acc_stride] : make_uint2(0u, 0u);
    const float2 ml0 = lane < n ? p.part_ml[base + (size_t)lane * p.R] : make_float2(-INFINITY, 0.f);
    float M = ml0.x;
    for (int c = lane + 32; c < n; c += 32) M = fmaxf(M, p.part_ml[base + (size_t)c * p.R].x);
    M = warp_max(M);
    const float w0 = ml0.y > 0.f ? ptx::ex2(ml0.x - M) * ml0.y : 0.f;
    float L = w0;
    for (int c = lane + 32; c < n; c += 32) {
      const float2 ml = p.part_ml[base + (size_t)c * p.R];
      if (ml.y > 0.f) L += ptx::ex2(ml.x - M) * ml.y;
    }
    L = warp_sum(L);
    // weight of split c (c is the same in every lane)
    auto weight = [&](int c) -> float {
      if (c < 32) return __shfl_sync(0xffffffffu, w0, c);
      const float2 ml = p.part_ml[base + (size_t)c * p.R];
      return ml.y > 0.f ? ptx::ex2(ml.x - M) * ml.y : 0.f;
    };
    auto add = [&](float w, const uint2& x) {
      const float2 v01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.x));
      const float2 v23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.y));
      o[0] += w * v01.x;
      o[1] += w * v01.y;
      o[2] += w * v23.x;
      o[3] += w * v23.y;
    };
#pragma unroll
    for (int c = 0; c < kPre; ++c) {
      const float w = weight(c);
      if (c < n) add(w, pre[c]);
    }
#pragma unroll 4
    for (int c = kPre; c < n; ++c) add(weight(c), acc[c * acc_stride]);
    const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] *= inv;
  }
  // n == 0: a refused sequence, its rows are zero
  uint2 w;
  w.x = pack_bf16(o[0], o[1]);
  w.y = pack_bf16(o[2], o[3]);
  reinterpret_cast<uint2*>(orow)[lane] = w;
}

// Persistent grid; each warp takes (pair, query row) units of the pairs the work list
// marked (split across items, or refused). Rows of whole-range items were written by
// the attention kernel. A marked pair's entry carries its item count.
__global__ void attn_combine_kernel(AttnTcParams p, const int* merge_list, const int* n_merge) {
  // the attention has read the old lengths: publish the lengths after the call
  if (blockIdx.x == 0 && p.lens)
    for (int b = threadIdx.x; b < p.batch; b += blockDim.x) p.lens[b] = p.lens_new[b];
  const int lane = threadIdx.x & 31;
  const int units = *n_merge * p.R;
  const int warps = gridDim.x * (blockDim.x >> 5);
  for (int u = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); u < units; u += warps) {
    const int e = merge_list[u / p.R];
    combine_row(p, e >> sched::kMergeCountShift, e & ((1 << sched::kMergeCountShift) - 1), u % p.R, lane);
  }
}

int sm_count() {
  static std::mutex mu;
  static int count[128] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 148;
  std::lock_guard<std::mutex> lock(mu);
  if (!count[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    count[dev] = n;
  }
  return count[dev];
}

template <bool NARROW, bool FP8>
cudaError_t launch_attn(const AttnTcParams& p, int grid, cudaStream_t s) {
  const size_t smem = Plan<NARROW, FP8>::SMEM;
  static_assert(Plan<NARROW, FP8>::SMEM <= 227 * 1024, "attention shared memory");
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<NARROW, FP8>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  LaunchScope ls_(DFLASH_KERNEL_ATTENTION, s);
  attn_tc_kernel<NARROW, FP8><<<grid, Plan<NARROW, FP8>::THREADS, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

// bf16 row-major [rows][cols] matrix, box {64, box_rows}, 128-byte swizzle (gemm_tc.cu)
bool encode_2d_bf16(CUtensorMap* m, const void* base, long long rows, int cols, int box_rows);
// byte matrix [rows][128], box {128, box_rows}, 128-byte swizzle (gemm_tc.cu)
bool encode_2d_u8(CUtensorMap* m, const void* base, long long rows, int box_rows);

int attn_tc_chunk() { return TK * sched::kItemMinTiles; }

// CTAs of the attention grid: one per SM (a work list covers at most sched::kMaxSm)
int attn_ctas() { return sm_count() < sched::kMaxSm ? sm_count() : sched::kMaxSm; }

size_t attn_sched_bytes(int batch, int n_kv) {
  return sched::area_bytes((size_t)batch * n_kv, (size_t)batch, (size_t)attn_ctas());
}

// Work-list buffers inside AttnParams::sched (sched::area_bytes): items [2 n_sm + pairs]
// int4, first [n_sm + 1], splits [pairs], 16 counters, qstart [batch], lens_new [batch],
// merge_list [pairs].
sched::Params attn_sched_params(const AttnParams& a) {
  const int pairs = a.batch * a.n_kv;
  const int n_sm = attn_ctas();
  sched::Params sp;
  sp.lens = a.lens;
  sp.pre_rows = a.pre_rows;
  sp.pre_M = a.pre_M;
  sp.items = (int4*)a.sched;
  sp.first = (int*)(sp.items + 2 * (size_t)n_sm + pairs);
  sp.splits = sp.first + n_sm + 1;
  sp.n_items = sp.splits + pairs;
  sp.n_merge = sp.n_items + 1;
  sp.ready = sp.n_items + 2;
  sp.qstart = sp.n_items + 16;
  sp.lens_new = sp.qstart + a.batch;
  sp.merge_list = sp.lens_new + a.batch;
  sp.batch = a.batch;
  sp.n_kv = a.n_kv;
  sp.bs = a.bs;
  sp.window = a.window;
  sp.capacity = a.capacity;
  sp.table_len = a.table_len;
  sp.max_splits = a.n_chunks;  // ranges are cut into at most this many items
  sp.n_sm = n_sm;
  sp.align = a.block_table ? TK : 1;
  // an item costs about 1.8 tiles of a CTA's time on a bf16 cache and 1.6 on E4M3 codes
  // (per-CTA timelines at the serving shape: the last tile's V load, the output stores,
  // the next item's first S)
  sp.item_cost = a.fp8 ? 13 : 14;
  return sp;
}

cudaError_t attn_worklist_build(const AttnParams& a, cudaStream_t s, sched::Params* sp) {
  *sp = attn_sched_params(a);
  LaunchScope ls_(DFLASH_KERNEL_SCHEDULE, s);
  attn_schedule_kernel<<<1, 1024, 0, s>>>(*sp);
  return cudaGetLastError();
}

cudaError_t attn_tc(const AttnParams& a, cudaStream_t s) {
  if (a.batch <= 0) return cudaSuccess;
  if (a.d_h != 128) return cudaErrorInvalidValue;
  // a merge-list entry packs the pair and its item count into one int
  if ((long long)a.batch * a.n_kv >= (1 << sched::kMergeCountShift) ||
      a.n_chunks >= (1 << (31 - sched::kMergeCountShift)))
    return cudaErrorInvalidValue;
  AttnTcParams p;
  memset(&p, 0, sizeof(p));
  const int R = (a.n_h / a.n_kv) * a.bs;
  const bool narrow = R <= 64;
  const long long kv_rows = a.block_table ? (long long)a.n_pages * a.n_kv * TK
                                          : (long long)a.batch * a.n_kv * a.capacity;
  const long long q_rows = (long long)a.batch * a.n_h * a.bs;
  if (a.fp8) {
    // Q codes, then the remainder codes, 128 bytes per row
    if (!encode_2d_u8(&p.q, a.q, q_rows, narrow ? 64 : 128) ||
        !encode_2d_u8(&p.q_lo, (const char*)a.q + q_rows * 128, q_rows, narrow ? 64 : 128) ||
        !encode_2d_u8(&p.k, a.cache_k, kv_rows, 128) || !encode_2d_u8(&p.v, a.cache_v, kv_rows, 128))
      return cudaErrorInvalidValue;
  } else if (!encode_2d_bf16(&p.q, a.q, q_rows, 128, narrow ? 64 : 128) ||
             !encode_2d_bf16(&p.k, a.cache_k, kv_rows, 128, 128) ||
             !encode_2d_bf16(&p.v, a.cache_v, kv_rows, 128, 128)) {
    return cudaErrorInvalidValue;
  }
  p.table = a.block_table;
  p.pps = a.pages_per_seq;
  const int pairs = a.batch * a.n_kv;
  const sched::Params sp = attn_sched_params(a);
  p.max_splits = sp.max_splits;
  p.qstart = sp.qstart;
  p.lens = a.lens_out;
  p.lens_new = sp.lens_new;
  p.out = (bf16*)a.out;
  p.out_v8 = ((uintptr_t)a.out & 31) == 0;
  p.part_acc = a.part_acc;
  p.part_ml = a.part_ml;
  p.items = sp.items;
  p.first = sp.first;
  p.status = a.status;
  p.batch = a.batch;
  p.n_h = a.n_h;
  p.n_kv = a.n_kv;
  p.bs = a.bs;
  p.G = a.n_h / a.n_kv;
  p.R = R;
  p.capacity = a.capacity;
  p.window = a.window;
  p.table_len = a.table_len;
  p.sl2 = a.scaling * 1.4426950408889634f * (a.fp8 ? a.k_scale : 1.f);
  p.v_scale = a.fp8 ? a.v_scale : 1.f;
  p.wait_ns = wait_limit_ns();
  p.list_ready = sp.ready;
  cudaError_t e = cudaSuccess;
  if (!a.sched_ready) {
    LaunchScope ls_(DFLASH_KERNEL_SCHEDULE, s);
    attn_schedule_kernel<<<1, 1024, 0, s>>>(sp);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return e;
  const int grid = sp.n_sm;  // the work list gives every SM a share (empty ones exit)
  if (a.fp8)
    e = narrow ? launch_attn<true, true>(p, grid, s) : launch_attn<false, true>(p, grid, s);
  else
    e = narrow ? launch_attn<true, false>(p, grid, s) : launch_attn<false, false>(p, grid, s);
  if (e != cudaSuccess) return e;
  // marked rows are at most pairs * R; a few waves of warps cover them
  const int rows = pairs * R;
  int cgrid = (rows + 7) / 8;
  if (cgrid > 4 * sp.n_sm) cgrid = 4 * sp.n_sm;
  LaunchScope ls_(DFLASH_KERNEL_COMBINE, s);
  attn_combine_kernel<<<cgrid, 256, 0, s>>>(p, sp.merge_list, sp.n_merge);
  return cudaGetLastError();
}

}  // namespace dflash
