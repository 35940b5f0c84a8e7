// Block attention on tcgen05 tensor cores (bf16 path).
//
// The G * bs queries of the block that share one KV head (G query heads x bs
// block positions, at most 128 rows) are stacked into one M=128 MMA tile, so
// every cached K/V row read from HBM serves all of them (DFlash KV Injection
// Walkthrough, Step 4.4: non-causal, every block query sees every key; DFlash
// source guide (II), part 1: query head h reads KV head h / G).
//
// Persistent kernel, one CTA per SM. Work items are (chunk, sequence, KV
// head) with chunks of 512 keys; CTAs take items round-robin. Per item:
//   warp 4      TMA producer: the Q tile once, then 128-key K and V tiles
//               into 2-stage rings (128-byte swizzle, L2 evict-first);
//   warp 5      MMA issuer: S_j = Q K_j^T into one of two TMEM S buffers,
//               O += P_j V_j into the TMEM O accumulator (V read MN-major);
//   warps 0-3   softmax, one thread per query row: masks the tile (chunk
//               end, sliding window), keeps a running max in the log2 domain,
//               rescales O in TMEM only when the max grows by more than 2^8,
//               writes P (bf16) into shared memory in the MMA's swizzled
//               layout, and at the end either writes out = O / l or, when
//               the sequence spans several chunks, a partial (m, l, O) that
//               the last CTA to finish that sequence and head merges.
#include <float.h>

#include <mutex>

#include "sm100_ptx.cuh"

namespace dflash {
namespace {

constexpr int TK = 128;                    // keys per tile
constexpr int CHUNK_TILES = 4;
constexpr int CHUNK = TK * CHUNK_TILES;    // keys per work item
constexpr int kThreads = 192;
constexpr uint32_t TILE = 128 * 128 * 2;   // 32 KB: Q, P, one K or one V tile
constexpr uint32_t HALF = TILE / 2;        // one 64-column swizzled box
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_P = TILE;
constexpr uint32_t OFF_K = 2 * TILE;       // 2 stages
constexpr uint32_t OFF_V = 4 * TILE;       // 2 stages
constexpr uint32_t OFF_BAR = 6 * TILE;
constexpr size_t SMEM = 1024 + OFF_BAR + 256 + 4096;  // slack past the barriers
constexpr uint32_t TM_S = 0, TM_O = 256;   // TMEM columns: S[2] at 0 and 128, O at 256
constexpr float kRescaleLog2 = 8.0f;       // rescale O only when the max grows by > 2^8

struct AttnTcParams {
  CUtensorMap q;   // [B*n_h*bs][128] bf16
  CUtensorMap k;   // [B*n_kv*capacity][128] bf16 (this layer)
  CUtensorMap v;
  const int32_t* lens;
  bf16* out;
  float* part_acc;
  float2* part_ml;
  int* counters;
  unsigned* status;
  int batch, n_h, n_kv, bs, G, R, capacity, window, table_len, max_chunks, total_items;
  float sl2;  // scaling * log2(e)
};

struct Item {
  int b, kvh, c, start, c0, c1, ntiles, nchunks;
  bool ok, valid;
};

__device__ __forceinline__ Item decode(const AttnTcParams& p, int i) {
  Item it;
  const int per = p.batch * p.n_kv;
  it.c = i / per;
  const int rem = i - it.c * per;
  it.b = rem / p.n_kv;
  it.kvh = rem - it.b * p.n_kv;
  it.start = p.lens[it.b];
  const int end = it.start + p.bs;
  const int lo = p.window > 0 ? max(0, it.start - p.window + 1) : 0;
  it.ok = it.start >= 0 && end <= p.capacity && end <= p.table_len;
  it.c0 = lo + it.c * CHUNK;
  it.c1 = min(end, it.c0 + CHUNK);
  it.valid = it.ok && it.c0 < it.c1;
  it.ntiles = it.valid ? (it.c1 - it.c0 + TK - 1) / TK : 0;
  it.nchunks = it.ok ? (end - lo + CHUNK - 1) / CHUNK : 0;
  return it;
}

__device__ __forceinline__ void drain(uint32_t bar, uint32_t parity, unsigned* status) {
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

template <bool DUP>
__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(const __grid_constant__ AttnTcParams p) {
  constexpr int NCOL = DUP ? 64 : 128;  // S columns per softmax thread
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(smem + OFF_BAR);
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ int last_flag;
  __shared__ float xch[2][2][64];  // DUP: tile maxima exchanged between the two column halves
  __shared__ float xl[2][64];      // DUP: row sums exchanged at the end of an item

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nsw = DUP ? 4 : (p.R + 31) >> 5;  // softmax warps holding query rows
  const uint32_t sbase = ptx::smem_u32(smem);
  // barriers
  const uint32_t q_full = ptx::smem_u32(bars + 0), q_empty = ptx::smem_u32(bars + 1);
  const uint32_t k_full0 = ptx::smem_u32(bars + 2), k_empty0 = ptx::smem_u32(bars + 4);
  const uint32_t v_full0 = ptx::smem_u32(bars + 6), v_empty0 = ptx::smem_u32(bars + 8);
  const uint32_t s_full0 = ptx::smem_u32(bars + 10), s_free0 = ptx::smem_u32(bars + 12);
  const uint32_t p_full = ptx::smem_u32(bars + 14), pv_done = ptx::smem_u32(bars + 15);

  if (threadIdx.x == 0) {
    abort_flag = 0;
    ptx::mbar_init(q_full, 1);
    ptx::mbar_init(q_empty, 1);
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(k_full0 + 8 * s, 1);
      ptx::mbar_init(k_empty0 + 8 * s, 1);
      ptx::mbar_init(v_full0 + 8 * s, 1);
      ptx::mbar_init(v_empty0 + 8 * s, 1);
      ptx::mbar_init(s_full0 + 8 * s, 1);
      ptx::mbar_init(s_free0 + 8 * s, 32 * nsw);
    }
    ptx::mbar_init(p_full, 32 * nsw);
    ptx::mbar_init(pv_done, 1);
    ptx::fence_mbar_init();
  }
  // P rows no softmax thread writes must hold zeros (finite) for the PV MMA
  {
    uint4* pz = reinterpret_cast<uint4*>(smem + OFF_P);
    for (int i = threadIdx.x; i < (int)(TILE / 16); i += blockDim.x) pz[i] = make_uint4(0, 0, 0, 0);
    ptx::fence_proxy_async_smem();
  }
  if (warp == 5) {
    ptx::tmem_alloc(ptx::smem_u32(&tmem_slot), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      ptx::prefetch_tmap(&p.q);
      ptx::prefetch_tmap(&p.k);
      ptx::prefetch_tmap(&p.v);
      const uint64_t pol = ptx::policy_evict_first();
      int gk = 0, gv = 0, n = 0;  // K tiles, V tiles, items issued
      bool stop = false;
      for (int i = blockIdx.x; i < p.total_items && !stop; i += gridDim.x) {
        const Item it = decode(p, i);
        if (!it.valid) continue;
        if (n > 0 && !ptx::mbar_wait(q_empty, (n - 1) & 1, &abort_flag, p.status)) break;
        const int qrow = (it.b * p.n_h + it.kvh * p.G) * p.bs;
        ptx::mbar_arrive_expect_tx(q_full, TILE);
        if (DUP) {  // 64 query rows, loaded twice: lanes 0-63 and 64-127
          ptx::tma_load_2d(sbase + OFF_Q, &p.q, q_full, 0, qrow);
          ptx::tma_load_2d(sbase + OFF_Q + 64 * 128, &p.q, q_full, 0, qrow);
          ptx::tma_load_2d(sbase + OFF_Q + HALF, &p.q, q_full, 64, qrow);
          ptx::tma_load_2d(sbase + OFF_Q + HALF + 64 * 128, &p.q, q_full, 64, qrow);
        } else {
          ptx::tma_load_2d(sbase + OFF_Q, &p.q, q_full, 0, qrow);
          ptx::tma_load_2d(sbase + OFF_Q + HALF, &p.q, q_full, 64, qrow);
        }
        ++n;
        const int kvrow = (it.b * p.n_kv + it.kvh) * p.capacity + it.c0;
        for (int j = 0; j < it.ntiles; ++j) {
          int s = gk & 1, u = gk >> 1;
          if (gk >= 2 && !ptx::mbar_wait(k_empty0 + 8 * s, (u - 1) & 1, &abort_flag, p.status)) {
            stop = true;
            break;
          }
          const uint32_t kd = sbase + OFF_K + s * TILE;
          ptx::mbar_arrive_expect_tx(k_full0 + 8 * s, TILE);
          ptx::tma_load_2d_hint(kd, &p.k, k_full0 + 8 * s, 0, kvrow + j * TK, pol);
          ptx::tma_load_2d_hint(kd + HALF, &p.k, k_full0 + 8 * s, 64, kvrow + j * TK, pol);
          ++gk;
          s = gv & 1;
          u = gv >> 1;
          if (gv >= 2 && !ptx::mbar_wait(v_empty0 + 8 * s, (u - 1) & 1, &abort_flag, p.status)) {
            stop = true;
            break;
          }
          const uint32_t vd = sbase + OFF_V + s * TILE;
          ptx::mbar_arrive_expect_tx(v_full0 + 8 * s, TILE);
          ptx::tma_load_2d_hint(vd, &p.v, v_full0 + 8 * s, 0, kvrow + j * TK, pol);
          ptx::tma_load_2d_hint(vd + HALF, &p.v, v_full0 + 8 * s, 64, kvrow + j * TK, pol);
          ++gv;
        }
      }
      // nothing of ours may still be landing in shared memory when the CTA exits
      if (n > 0) drain(q_full, (n - 1) & 1, p.status);
      for (int g = gk > 2 ? gk - 2 : 0; g < gk; ++g) drain(k_full0 + 8 * (g & 1), (g >> 1) & 1, p.status);
      for (int g = gv > 2 ? gv - 2 : 0; g < gv; ++g) drain(v_full0 + 8 * (g & 1), (g >> 1) & 1, p.status);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = ptx::idesc_bf16_f32(128, TK);
      constexpr uint32_t idesc_pv = ptx::idesc_bf16_f32(128, 128) | (1u << 16);  // B (V) MN-major
      int gt = 0, n = 0;
      bool stop = false;
      for (int i = blockIdx.x; i < p.total_items && !stop; i += gridDim.x) {
        const Item it = decode(p, i);
        if (!it.valid) continue;
        if (!ptx::mbar_wait(q_full, n & 1, &abort_flag, p.status)) break;
        const int T = it.ntiles, base = gt;
        auto issue_s = [&](int j) -> bool {
          const int g = base + j, s = g & 1, u = g >> 1;
          if (g >= 2 && !ptx::mbar_wait(s_free0 + 8 * s, (u - 1) & 1, &abort_flag, p.status))
            return false;
          if (!ptx::mbar_wait(k_full0 + 8 * s, u & 1, &abort_flag, p.status)) return false;
          ptx::tc_fence_after();
          const uint32_t qa = sbase + OFF_Q, ka = sbase + OFF_K + s * TILE;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * HALF + (kk & 3) * 32;
            ptx::mma_bf16(tmem + TM_S + s * TK, ptx::smem_desc_sw128(qa + off),
                          ptx::smem_desc_sw128(ka + off), idesc_s, kk > 0 ? 1u : 0u);
          }
          ptx::mma_commit(k_empty0 + 8 * s);
          ptx::mma_commit(s_full0 + 8 * s);
          if (j == T - 1) ptx::mma_commit(q_empty);
          return true;
        };
        if (!issue_s(0) || (T > 1 && !issue_s(1))) break;
        for (int j = 0; j < T; ++j) {
          const int g = base + j, s = g & 1, u = g >> 1;
          if (!ptx::mbar_wait(p_full, g & 1, &abort_flag, p.status) ||
              !ptx::mbar_wait(v_full0 + 8 * s, u & 1, &abort_flag, p.status)) {
            stop = true;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t pa = sbase + OFF_P, va = sbase + OFF_V + s * TILE;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            ptx::mma_bf16(tmem + TM_O,
                          ptx::smem_desc_sw128(pa + (kk >> 2) * HALF + (kk & 3) * 32),
                          ptx::smem_desc_sw128_mn(va + kk * 2048, HALF), idesc_pv,
                          (j > 0 || kk > 0) ? 1u : 0u);
          ptx::mma_commit(v_empty0 + 8 * s);
          ptx::mma_commit(pv_done);
          if (j + 2 < T && !issue_s(j + 2)) {
            stop = true;
            break;
          }
        }
        gt = base + T;
        ++n;
      }
      // every MMA has finished before TMEM is released
      if (gt > 0) drain(pv_done, (gt - 1) & 1, p.status);
    }
  } else if (warp < nsw) {
    // ------------------------------------------------------------ softmax rows
    // DUP: the query rows fill TMEM lanes 0-63 and again 64-127; warps 0-1 take
    // columns 0-63 of each row and warps 2-3 columns 64-127, and exchange the tile
    // maximum and the final row sum through shared memory.
    const int rt = warp * 32 + lane;                 // TMEM lane = S / O row
    const int qr = DUP ? (rt & 63) : rt;             // query row (g * bs + t)
    const int half = DUP ? (warp >> 1) : 0;
    const int coff = half * NCOL;                    // first column this thread owns
    const bool rvalid = qr < p.R;
    const int gq = rvalid ? qr / p.bs : 0, t = rvalid ? qr - gq * p.bs : 0;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const uint32_t nsync = 32 * nsw;
    uint8_t* pbase = smem + OFF_P;
    int gt = 0;
    float s[NCOL];
    for (int i = blockIdx.x; i < p.total_items; i += gridDim.x) {
      const Item it = decode(p, i);
      if (!it.ok) {
        // a refused sequence (capacity / table): its output rows are zero
        if (it.c == 0 && rvalid) {
          uint4* o = reinterpret_cast<uint4*>(p.out + ((size_t)(it.b * p.bs + t) * p.n_h +
                                                       it.kvh * p.G + gq) * 128 + coff);
          for (int k = 0; k < NCOL / 8; ++k) o[k] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      if (!it.valid) continue;
      const int T = it.ntiles;
      const int qpos = it.start + t;
      float m_ref = -INFINITY, l = 0.f;
      bool alive = true;
      for (int j = 0; j < T && alive; ++j) {
        const int g = gt + j, sb = g & 1, u = g >> 1;
        alive = __all_sync(0xffffffffu, ptx::mbar_wait(s_full0 + 8 * sb, u & 1, &abort_flag, p.status));
        if (!alive) break;
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
        const int key0 = it.c0 + j * TK + coff;
        const bool full = rvalid && key0 + NCOL <= it.c1 && (p.window <= 0 || qpos - key0 < p.window);
        float mx;
        if (full) {
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int e = 0; e < NCOL; ++e) m4[e & 3] = fmaxf(m4[e & 3], s[e]);
          mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        } else {
          mx = -INFINITY;
#pragma unroll
          for (int e = 0; e < NCOL; ++e) {
            const int key = key0 + e;
            const bool vis = rvalid && key < it.c1 && (p.window <= 0 || qpos - key < p.window);
            s[e] = vis ? s[e] : -INFINITY;
            mx = fmaxf(mx, s[e]);
          }
        }
        if (DUP) {
          xch[j & 1][half][qr] = mx;
          ptx::named_sync(2, nsync);
          mx = fmaxf(mx, xch[j & 1][half ^ 1][qr]);
        }
        mx *= p.sl2;  // log2 domain
        float alpha = 1.f;
        bool resc = false;
        if (m_ref == -INFINITY) {
          m_ref = mx;                      // nothing accumulated yet for this row
        } else if (mx > m_ref + kRescaleLog2) {
          alpha = ptx::ex2(m_ref - mx);
          m_ref = mx;
          resc = true;
        }
        const float mu = (m_ref == -INFINITY) ? 0.f : m_ref;
        const float2 sl2v = make_float2(p.sl2, p.sl2), nmu = make_float2(-mu, -mu);
        float2 acc2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                          make_float2(0.f, 0.f)};
#pragma unroll
        for (int e = 0; e < NCOL; e += 2) {
          const float2 x = __ffma2_rn(make_float2(s[e], s[e + 1]), sl2v, nmu);
          s[e] = ptx::ex2(x.x);
          s[e + 1] = ptx::ex2(x.y);
          acc2[(e >> 1) & 3] = __fadd2_rn(acc2[(e >> 1) & 3], make_float2(s[e], s[e + 1]));
        }
        const float2 a01 = __fadd2_rn(acc2[0], acc2[1]), a23 = __fadd2_rn(acc2[2], acc2[3]);
        l = l * alpha + ((a01.x + a01.y) + (a23.x + a23.y));
        if (j > 0) {
          // PV of the previous tile done: P may be overwritten, O holds tiles < j
          alive = __all_sync(0xffffffffu, ptx::mbar_wait(pv_done, (g - 1) & 1, &abort_flag, p.status));
          if (!alive) break;
          ptx::tc_fence_after();
          if (__any_sync(0xffffffffu, resc)) {
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
        }
        // P, bf16, in the 128-byte-swizzled K-major layout the MMA reads: this thread's
        // keys coff .. coff+NCOL-1 of query row qr (and of its copy qr + 64 under DUP)
#pragma unroll
        for (int cidx = 0; cidx < NCOL / 8; ++cidx) {
          const int key = coff + 8 * cidx, kb = key >> 6, cc = (key >> 3) & 7;
          uint4 w;
          w.x = pack_bf16(s[8 * cidx + 0], s[8 * cidx + 1]);
          w.y = pack_bf16(s[8 * cidx + 2], s[8 * cidx + 3]);
          w.z = pack_bf16(s[8 * cidx + 4], s[8 * cidx + 5]);
          w.w = pack_bf16(s[8 * cidx + 6], s[8 * cidx + 7]);
          *reinterpret_cast<uint4*>(pbase + kb * HALF + qr * 128 + ((cc ^ (qr & 7)) << 4)) = w;
          if (DUP)
            *reinterpret_cast<uint4*>(pbase + kb * HALF + (qr + 64) * 128 + ((cc ^ (qr & 7)) << 4)) = w;
        }
        // keys past the chunk end in the last tile: zero their V rows (slots past the
        // cache length may hold anything, and 0 * NaN would poison O)
        const int nvalid = it.c1 - (it.c0 + j * TK);
        if (j == T - 1 && nvalid < TK) {
          alive = __all_sync(0xffffffffu, ptx::mbar_wait(v_full0 + 8 * sb, u & 1, &abort_flag, p.status));
          if (!alive) break;
          uint4* vz = reinterpret_cast<uint4*>(smem + OFF_V + sb * TILE);
          const int per_half = (TK - nvalid) * 8;  // 16-byte chunks per half
          for (int idx = rt; idx < 2 * per_half; idx += nsync) {
            const int h = idx / per_half, rem = idx - h * per_half;
            vz[(h * HALF) / 16 + nvalid * 8 + rem] = make_uint4(0, 0, 0, 0);
          }
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        ptx::mbar_arrive(p_full);
      }
      if (!alive) break;
      gt += T;
      // ---- epilogue: this thread's columns of O for this item
      if (DUP) {
        // row sum of both halves; the barrier also ends every read of xch for this item
        xl[half][qr] = l;
        ptx::named_sync(2, nsync);
        l += xl[half ^ 1][qr];
      }
      alive = __all_sync(0xffffffffu, ptx::mbar_wait(pv_done, (gt - 1) & 1, &abort_flag, p.status));
      if (!alive) break;
      ptx::tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < NCOL / 32; ++cc) {
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(tmem + lane_base + TM_O + coff + cc * 32, v);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) s[cc * 32 + e] = __uint_as_float(v[e]);
      }
      const int bk = it.b * p.n_kv + it.kvh;
      bf16* orow = p.out + ((size_t)(it.b * p.bs + t) * p.n_h + it.kvh * p.G + gq) * 128 + coff;
      if (it.nchunks == 1) {
        if (rvalid) {
          const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
          for (int k = 0; k < NCOL / 8; ++k) {
            uint4 w;
            w.x = pack_bf16(s[8 * k + 0] * inv, s[8 * k + 1] * inv);
            w.y = pack_bf16(s[8 * k + 2] * inv, s[8 * k + 3] * inv);
            w.z = pack_bf16(s[8 * k + 4] * inv, s[8 * k + 5] * inv);
            w.w = pack_bf16(s[8 * k + 6] * inv, s[8 * k + 7] * inv);
            reinterpret_cast<uint4*>(orow)[k] = w;
          }
        }
        continue;
      }
      // several chunks: publish this chunk's partial, the last one merges
      const size_t prow_idx = ((size_t)bk * p.max_chunks + it.c) * p.R + qr;
      if (rvalid) {
        float4* a = reinterpret_cast<float4*>(p.part_acc + prow_idx * 128 + coff);
#pragma unroll
        for (int k = 0; k < NCOL / 4; ++k) a[k] = make_float4(s[4 * k], s[4 * k + 1], s[4 * k + 2], s[4 * k + 3]);
        if (half == 0) p.part_ml[prow_idx] = make_float2(m_ref, l);
      }
      __threadfence();
      ptx::named_sync(1, nsync);
      if (threadIdx.x == 0) last_flag = (atomicAdd(p.counters + bk, 1) == it.nchunks - 1);
      ptx::named_sync(1, nsync);
      if (!last_flag) continue;
      __threadfence();
      if (rvalid) {
        const size_t base = (size_t)bk * p.max_chunks * p.R + qr;
        float M = -INFINITY;
        for (int c = 0; c < it.nchunks; ++c) M = fmaxf(M, __ldcg(p.part_ml + base + (size_t)c * p.R).x);
        float L = 0.f;
        float acc[NCOL];
#pragma unroll
        for (int e = 0; e < NCOL; ++e) acc[e] = 0.f;
        for (int c = 0; c < it.nchunks; ++c) {
          const float2 ml = __ldcg(p.part_ml + base + (size_t)c * p.R);
          if (ml.y == 0.f) continue;
          const float w = ptx::ex2(ml.x - M);
          L += w * ml.y;
          const float4* a = reinterpret_cast<const float4*>(p.part_acc + (base + (size_t)c * p.R) * 128 + coff);
#pragma unroll
          for (int k = 0; k < NCOL / 4; ++k) {
            const float4 x = __ldcg(a + k);
            acc[4 * k] += w * x.x;
            acc[4 * k + 1] += w * x.y;
            acc[4 * k + 2] += w * x.z;
            acc[4 * k + 3] += w * x.w;
          }
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
        for (int k = 0; k < NCOL / 8; ++k) {
          uint4 w;
          w.x = pack_bf16(acc[8 * k + 0] * inv, acc[8 * k + 1] * inv);
          w.y = pack_bf16(acc[8 * k + 2] * inv, acc[8 * k + 3] * inv);
          w.z = pack_bf16(acc[8 * k + 4] * inv, acc[8 * k + 5] * inv);
          w.w = pack_bf16(acc[8 * k + 6] * inv, acc[8 * k + 7] * inv);
          reinterpret_cast<uint4*>(orow)[k] = w;
        }
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// ---- host side ---------------------------------------------------------------

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

}  // namespace

// bf16 row-major [rows][cols] matrix, box {64, box_rows}, 128-byte swizzle (gemm_tc.cu)
bool encode_2d_bf16(CUtensorMap* m, const void* base, long long rows, int cols, int box_rows);

int attn_tc_chunk() { return CHUNK; }

cudaError_t attn_tc(const AttnParams& a, cudaStream_t s) {
  if (a.batch <= 0) return cudaSuccess;
  if (a.d_h != 128) return cudaErrorInvalidValue;
  AttnTcParams p;
  memset(&p, 0, sizeof(p));
  const int R = (a.n_h / a.n_kv) * a.bs;
  const bool dup = R <= 64;
  if (!encode_2d_bf16(&p.q, a.q, (long long)a.batch * a.n_h * a.bs, 128, dup ? 64 : 128) ||
      !encode_2d_bf16(&p.k, a.cache_k, (long long)a.batch * a.n_kv * a.capacity, 128, 128) ||
      !encode_2d_bf16(&p.v, a.cache_v, (long long)a.batch * a.n_kv * a.capacity, 128, 128))
    return cudaErrorInvalidValue;
  p.lens = a.lens;
  p.out = (bf16*)a.out;
  p.part_acc = a.part_acc;
  p.part_ml = a.part_ml;
  p.counters = a.counters;
  p.status = a.status;
  p.batch = a.batch;
  p.n_h = a.n_h;
  p.n_kv = a.n_kv;
  p.bs = a.bs;
  p.G = a.n_h / a.n_kv;
  p.R = p.G * a.bs;
  p.capacity = a.capacity;
  p.window = a.window;
  p.table_len = a.table_len;
  p.max_chunks = a.n_chunks;
  p.total_items = a.n_chunks * a.batch * a.n_kv;
  p.sl2 = a.scaling * 1.4426950408889634f;
  cudaError_t e = cudaMemsetAsync(a.counters, 0, sizeof(int) * a.batch * a.n_kv, s);
  if (e != cudaSuccess) return e;
  int grid = sm_count();
  if (grid > p.total_items) grid = p.total_items;
  if (dup) {
    e = cudaFuncSetAttribute(attn_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM);
    if (e != cudaSuccess) return e;
    LaunchScope ls_(DFLASH_KERNEL_ATTENTION, s);
    attn_tc_kernel<true><<<grid, kThreads, SMEM, s>>>(p);
  } else {
    e = cudaFuncSetAttribute(attn_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM);
    if (e != cudaSuccess) return e;
    LaunchScope ls_(DFLASH_KERNEL_ATTENTION, s);
    attn_tc_kernel<false><<<grid, kThreads, SMEM, s>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace dflash
