// SIMT split-KV block attention (the fp32 path).
//
// Non-causal attention of the block's bs queries of one head over the
// cached rows [lo, start + bs) of its KV head (DFlash KV Injection
// Walkthrough, Step 4.4; DFlash source guide (II), non-causal design note
// and part 5 for the sliding window). Keys are cut into chunks; each CTA
// runs an online softmax over one chunk and leaves an un-normalised partial
// (running max m, running sum l, accumulator acc), and the combine kernel
// merges the chunks with the usual log-sum-exp rescaling.
#include <float.h>

#include "dflash_internal.cuh"

namespace dflash {
namespace {

constexpr int CHUNK = 256;   // keys per CTA
constexpr int TILE = 32;     // keys staged in shared memory at a time
constexpr int MAXD = 8;      // d_h / 32 elements of the accumulator per lane (d_h <= 256)
constexpr int MAXQ = 4;      // queries per warp (bs <= 16 with 4 warps)

struct Range { int start, end, lo; };

__device__ __forceinline__ Range key_range(const AttnParams& p, int b) {
  Range r;
  r.start = p.lens[b];
  r.end = r.start + p.bs;
  r.lo = 0;
  if (p.window > 0) r.lo = max(0, r.start - p.window + 1);
  return r;
}

__device__ __forceinline__ bool range_ok(const AttnParams& p, const Range& r) {
  return r.start >= 0 && r.end <= p.capacity && r.end <= p.table_len;
}

template <typename T>
__global__ void __launch_bounds__(128) attn_simt_kernel(AttnParams p) {
  extern __shared__ float smem[];
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int G = p.n_h / p.n_kv, kvh = h / G, dh = p.d_h;
  const int ld = dh + 1;
  float* q_s = smem;                  // [bs][dh]
  float* k_s = q_s + p.bs * dh;       // [TILE][dh + 1]
  float* v_s = k_s + TILE * ld;       // [TILE][dh]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const Range r = key_range(p, b);
  const bool ok = range_ok(p, r);
  const int c0 = r.lo + c * p.chunk;
  const int c1 = min(r.end, c0 + p.chunk);
  const size_t part = (((size_t)b * p.n_h + h) * p.n_chunks + c) * p.bs;

  float m[MAXQ], l[MAXQ], acc[MAXQ][MAXD];
#pragma unroll
  for (int i = 0; i < MAXQ; ++i) {
    m[i] = -FLT_MAX;
    l[i] = 0.f;
#pragma unroll
    for (int j = 0; j < MAXD; ++j) acc[i][j] = 0.f;
  }

  if (ok && c0 < c1) {
    const T* q = (const T*)p.q + ((size_t)b * p.n_h + h) * p.bs * dh;
    for (int e = threadIdx.x; e < p.bs * dh; e += blockDim.x) q_s[e] = to_f(q[e]) * p.scaling;
    const size_t kvbase = ((size_t)b * p.n_kv + kvh) * p.capacity;
    const T* K = (const T*)p.cache_k + kvbase * dh;
    const T* V = (const T*)p.cache_v + kvbase * dh;
    for (int j0 = c0; j0 < c1; j0 += TILE) {
      const int nt = min(TILE, c1 - j0);
      __syncthreads();
      for (int e = threadIdx.x; e < nt * dh; e += blockDim.x) {
        const int jj = e / dh, dd = e - jj * dh;
        k_s[jj * ld + dd] = to_f(K[(size_t)(j0 + jj) * dh + dd]);
        v_s[jj * dh + dd] = to_f(V[(size_t)(j0 + jj) * dh + dd]);
      }
      __syncthreads();
#pragma unroll
      for (int qi = 0; qi < MAXQ; ++qi) {
        const int t = warp + 4 * qi;
        if (t >= p.bs) break;
        const int qpos = r.start + t;
        // lane owns key j0 + lane
        float s = -FLT_MAX;
        const int j = j0 + lane;
        if (lane < nt && (p.window <= 0 || qpos - j < p.window)) {
          float dot = 0.f;
          const float* qq = q_s + t * dh;
          const float* kk = k_s + lane * ld;
          for (int dd = 0; dd < dh; ++dd) dot = fmaf(qq[dd], kk[dd], dot);
          s = dot;
        }
        const float mt = warp_max(s);
        if (mt == -FLT_MAX) continue;  // no visible key in this tile for this query
        const float mn = fmaxf(m[qi], mt);
        const float corr = expf(m[qi] - mn);
        const float pl = (s == -FLT_MAX) ? 0.f : expf(s - mn);
        l[qi] = l[qi] * corr + warp_sum(pl);
        m[qi] = mn;
#pragma unroll
        for (int dd = 0; dd < MAXD; ++dd) acc[qi][dd] *= corr;
        for (int jj = 0; jj < nt; ++jj) {
          const float pj = __shfl_sync(0xffffffffu, pl, jj);
#pragma unroll
          for (int dd = 0; dd < MAXD; ++dd) {
            const int col = lane + 32 * dd;
            if (col < dh) acc[qi][dd] = fmaf(pj, v_s[jj * dh + col], acc[qi][dd]);
          }
        }
      }
    }
  }
  // write the partial, or the final row when the whole range is one chunk
#pragma unroll
  for (int qi = 0; qi < MAXQ; ++qi) {
    const int t = warp + 4 * qi;
    if (t >= p.bs) break;
    if (p.n_chunks == 1) {
      T* o = (T*)p.out + ((size_t)b * p.bs + t) * p.n_h * dh + (size_t)h * dh;
      const float inv = (ok && l[qi] > 0.f) ? 1.0f / l[qi] : 0.f;
#pragma unroll
      for (int dd = 0; dd < MAXD; ++dd) {
        const int col = lane + 32 * dd;
        if (col < dh) o[col] = from_f<T>(acc[qi][dd] * inv);
      }
    } else {
      float* a = p.part_acc + (part + t) * dh;
#pragma unroll
      for (int dd = 0; dd < MAXD; ++dd) {
        const int col = lane + 32 * dd;
        if (col < dh) a[col] = acc[qi][dd];
      }
      if (lane == 0) p.part_ml[part + t] = make_float2(m[qi], l[qi]);
    }
  }
}

// One warp per output row (b, t, h): merge the chunks' partials.
template <typename T>
__global__ void attn_combine_kernel(AttnParams p) {
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= p.batch * p.n_h * p.bs) return;
  const int t = row % p.bs, h = (row / p.bs) % p.n_h, b = row / (p.bs * p.n_h);
  const int dh = p.d_h;
  const Range r = key_range(p, b);
  T* o = (T*)p.out + ((size_t)b * p.bs + t) * p.n_h * dh + (size_t)h * dh;
  if (!range_ok(p, r)) {
    for (int col = lane; col < dh; col += 32) o[col] = from_f<T>(0.f);
    return;
  }
  const int nc = min(p.n_chunks, (r.end - r.lo + p.chunk - 1) / p.chunk);
  const size_t part = ((size_t)b * p.n_h + h) * p.n_chunks;
  float M = -FLT_MAX;
  for (int c = 0; c < nc; ++c) M = fmaxf(M, p.part_ml[(part + c) * p.bs + t].x);
  float L = 0.f;
  float acc[MAXD] = {};
  for (int c = 0; c < nc; ++c) {
    const float2 ml = p.part_ml[(part + c) * p.bs + t];
    if (ml.y == 0.f) continue;
    const float w = expf(ml.x - M);
    L += w * ml.y;
    const float* a = p.part_acc + ((part + c) * p.bs + t) * dh;
#pragma unroll
    for (int dd = 0; dd < MAXD; ++dd) {
      const int col = lane + 32 * dd;
      if (col < dh) acc[dd] = fmaf(w, a[col], acc[dd]);
    }
  }
  const float inv = L > 0.f ? 1.0f / L : 0.f;
#pragma unroll
  for (int dd = 0; dd < MAXD; ++dd) {
    const int col = lane + 32 * dd;
    if (col < dh) o[col] = from_f<T>(acc[dd] * inv);
  }
}

}  // namespace

int attn_simt_chunk() { return CHUNK; }

cudaError_t attn_simt(int dtype, const AttnParams& p, cudaStream_t s) {
  if (p.batch <= 0) return cudaSuccess;
  dim3 grid(p.n_chunks, p.n_h, p.batch);
  const size_t sm = (size_t)(p.bs * p.d_h + TILE * (p.d_h + 1) + TILE * p.d_h) * sizeof(float);
  if (dtype == DFLASH_F32) {
    if (sm > 48 * 1024)
      cudaFuncSetAttribute(attn_simt_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)sm);
    {
      LaunchScope ls_(DFLASH_KERNEL_ATTENTION, s);
      attn_simt_kernel<float><<<grid, 128, sm, s>>>(p);
    }
  } else {
    if (sm > 48 * 1024)
      cudaFuncSetAttribute(attn_simt_kernel<bf16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)sm);
    {
      LaunchScope ls_(DFLASH_KERNEL_ATTENTION, s);
      attn_simt_kernel<bf16><<<grid, 128, sm, s>>>(p);
    }
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.n_chunks == 1) return e;
  const int rows = p.batch * p.n_h * p.bs;
  if (dtype == DFLASH_F32)
    {
      LaunchScope ls_(DFLASH_KERNEL_COMBINE, s);
      attn_combine_kernel<float><<<(rows + 3) / 4, 128, 0, s>>>(p);
    }
  else
    {
      LaunchScope ls_(DFLASH_KERNEL_COMBINE, s);
      attn_combine_kernel<bf16><<<(rows + 3) / 4, 128, 0, s>>>(p);
    }
  return cudaGetLastError();
}

}  // namespace dflash
