// Row-wise epilogues, cache bookkeeping and the RoPE table.
//
//  - rmsnorm_rows: hidden_norm of the context signal (DFlash KV Injection
//    Walkthrough, Step 2).
//  - head_epilogue: per-head QNorm / KNorm, RoPE at absolute positions and
//    the scatter of K/V rows into the draft cache (Steps 4.1-4.3; DFlash
//    source guide (II), parts 1-4).
//  - lens_advance / crop_lens: the cache's update() length bump and
//    crop(start) (source guide part 4; walkthrough Step 7).
//  - rope_table: cos/sin of p * theta^(-2i/d_h) in double precision.
#include "attn_sched.cuh"

namespace dflash {
namespace {

__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31, nw = (blockDim.x + 31) >> 5;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float t = 0.f;
  for (int i = 0; i < nw; ++i) t += red[i];
  return t;
}

template <typename T>
__global__ void rmsnorm_rows_kernel(const float* __restrict__ Y, int splits, int M, int N,
                                    const T* __restrict__ gamma, float eps, T* __restrict__ out) {
  __shared__ float red[32];
  const int row = blockIdx.x;
  const size_t split_stride = (size_t)M * N;
  float ss = 0.f;
  for (int c = threadIdx.x; c < N; c += blockDim.x) {
    float y = 0.f;
    for (int s = 0; s < splits; ++s) y += Y[s * split_stride + (size_t)row * N + c];
    ss += y * y;
  }
  ss = block_sum(ss, red);
  const float r = 1.0f / sqrtf(ss / (float)N + eps);
  for (int c = threadIdx.x; c < N; c += blockDim.x) {
    float y = 0.f;
    for (int s = 0; s < splits; ++s) y += Y[s * split_stride + (size_t)row * N + c];
    out[(size_t)row * N + c] = from_f<T>(y * r * to_f(gamma[c]));
  }
}

// Single pass: each thread keeps its float4 chunks of the row (summed over the
// splits) in registers, one block reduction, then scale and store. N <= 8192.
constexpr int kNormThreads = 256, kNormMaxChunks = 8;

template <typename T>
__device__ __forceinline__ void store4(T* dst, float4 v);
template <>
__device__ __forceinline__ void store4<float>(float* dst, float4 v) {
  *reinterpret_cast<float4*>(dst) = v;
}
template <>
__device__ __forceinline__ void store4<bf16>(bf16* dst, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(dst) = u;
}

// v[k] = sum over the splits of chunk k (thread's columns 4 (threadIdx.x + k NT)), added
// in pairs of consecutive splits; the loads of SB splits (an even count) are issued
// before any of them is added, so a row costs one memory round trip per SB splits.
template <int CH, int NT, int SB>
__device__ __forceinline__ void sum_splits(const float4* __restrict__ y4, size_t split_stride4,
                                           int splits, int n4, float4 (&v)[CH]) {
  static_assert(SB % 2 == 0, "splits are added in pairs");
#pragma unroll
  for (int k = 0; k < CH; ++k) v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < splits; s0 += SB) {
    float4 a[SB][CH];
#pragma unroll
    for (int j = 0; j < SB; ++j)
#pragma unroll
      for (int k = 0; k < CH; ++k) {
        const int c = threadIdx.x + k * NT;
        a[j][k] = (s0 + j < splits && c < n4) ? y4[(s0 + j) * split_stride4 + c]
                                              : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
    for (int j = 0; j < SB; j += 2)
#pragma unroll
      for (int k = 0; k < CH; ++k) {
        v[k].x += a[j][k].x + a[j + 1][k].x;
        v[k].y += a[j][k].y + a[j + 1][k].y;
        v[k].z += a[j][k].z + a[j + 1][k].z;
        v[k].w += a[j][k].w + a[j + 1][k].w;
      }
  }
}

template <typename T>
__device__ __forceinline__ float4 load_gamma4(const T* g) {
  return make_float4(to_f(g[0]), to_f(g[1]), to_f(g[2]), to_f(g[3]));
}
template <>
__device__ __forceinline__ float4 load_gamma4<bf16>(const bf16* g) {
  const uint2 u = *reinterpret_cast<const uint2*>(g);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

// One CTA of NT threads per row; chunk k of a thread is float4 column threadIdx.x + k NT.
template <typename T, int CH, int NT>
__global__ void __launch_bounds__(NT) rmsnorm_rows_vec_kernel(
    const float* __restrict__ Y, int splits, int M, int N, const T* __restrict__ gamma, float eps,
    T* __restrict__ out) {
  __shared__ float red[32];
  const int row = blockIdx.x;
  const int n4 = N >> 2;
  const size_t split_stride4 = (size_t)M * n4;
  const float4* y4 = reinterpret_cast<const float4*>(Y) + (size_t)row * n4;
  float4 g[CH];
#pragma unroll
  for (int k = 0; k < CH; ++k) {
    const int c = threadIdx.x + k * NT;
    g[k] = c < n4 ? load_gamma4(gamma + 4 * c) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float4 v[CH];
  sum_splits<CH, NT, (CH <= 2 ? 8 : 2)>(y4, split_stride4, splits, n4, v);
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < CH; ++k)
    ss += v[k].x * v[k].x + v[k].y * v[k].y + v[k].z * v[k].z + v[k].w * v[k].w;
  ss = block_sum(ss, red);
  const float r = 1.0f / sqrtf(ss / (float)N + eps);
#pragma unroll
  for (int k = 0; k < CH; ++k) {
    const int c = threadIdx.x + k * NT;
    if (c < n4)
      store4<T>(out + (size_t)row * N + 4 * c, make_float4(v[k].x * r * g[k].x, v[k].y * r * g[k].y,
                                                           v[k].z * r * g[k].z, v[k].w * r * g[k].w));
  }
}

// One CTA per (row, head); thread i handles the RoPE pair (i, i + d_h/2).
template <typename T>
__global__ void head_epilogue_kernel(HeadEpilogue e) {
  __shared__ float red[32];
  const int row = blockIdx.y, head = blockIdx.x;
  const int half = e.d_h / 2;
  // row -> (sequence, index within its rows)
  int b, t, n_b;
  if (e.cu_rows) {
    int lo = 0, hi = e.batch - 1;
    while (lo < hi) {  // last b with cu_rows[b] <= row
      int mid = (lo + hi + 1) >> 1;
      if (e.cu_rows[mid] <= row) lo = mid; else hi = mid - 1;
    }
    b = lo;
    t = row - e.cu_rows[b];
    n_b = e.cu_rows[b + 1] - e.cu_rows[b];
    if (n_b < 0 || e.cu_rows[b + 1] > e.rows || e.cu_rows[0] != 0 || t < 0 || t >= n_b) {
      if (threadIdx.x == 0) atomicOr(e.status, DFLASH_DEV_ROWS);
      return;
    }
  } else {
    b = row / e.bs;
    t = row - b * e.bs;
    n_b = e.bs;
  }
  int start = e.lens[b];
  start += sched::injected_rows(e.pre_rows, e.pre_M, b, start, e.capacity, e.table_len);
  const int pos = start + t;
  if (start < 0 || start + n_b > e.capacity || start + n_b > e.table_len) {
    if (threadIdx.x == 0 && t == 0 && head == 0)
      atomicOr(e.status, (start + n_b > e.capacity || start < 0) ? DFLASH_DEV_CAPACITY
                                                                 : DFLASH_DEV_ROPE);
    return;
  }
  const size_t split_stride = (size_t)e.rows * e.ldY;
  const float* y = e.Y + (size_t)row * e.ldY + (size_t)head * e.d_h;
  const int i = threadIdx.x;
  float x0 = 0.f, x1 = 0.f;
  if (i < half) {
    for (int s = 0; s < e.splits; ++s) {
      x0 += y[s * split_stride + i];
      x1 += y[s * split_stride + i + half];
    }
  }
  const int kind = head < e.n_q ? 0 : (head < e.n_q + e.n_kv ? 1 : 2);  // Q, K, V
  if (kind < 2) {
    const float ss = block_sum(x0 * x0 + x1 * x1, red);
    const float r = 1.0f / sqrtf(ss / (float)e.d_h + e.eps);
    const T* g = (const T*)(kind == 0 ? e.gamma_q : e.gamma_k);
    if (i < half) {
      x0 = x0 * r * to_f(g[i]);
      x1 = x1 * r * to_f(g[i + half]);
      const float2 cs = e.rope[(size_t)pos * half + i];
      const float r0 = x0 * cs.x - x1 * cs.y;  // rotate_half: [-x1, x0]
      const float r1 = x1 * cs.x + x0 * cs.y;
      x0 = r0;
      x1 = r1;
    }
  }
  if (i >= half) return;
  T* dst;
  if (kind == 0) {
    dst = (T*)e.q_out + (((size_t)b * e.n_q + head) * e.bs + t) * e.d_h;
  } else {
    const int kvh = head - e.n_q - (kind == 2 ? e.n_kv : 0);
    T* base = (T*)(kind == 1 ? e.cache_k : e.cache_v);
    dst = base + cache_row(e.block_table, e.pages_per_seq, e.n_kv, e.capacity, b, kvh, pos) * e.d_h;
  }
  dst[i] = from_f<T>(x0);
  dst[i + half] = from_f<T>(x1);
}

// bf16, d_h = 128: one warp per (row, head); lane l holds dims 4l .. 4l+3, so the
// RoPE partner (i + 64) of lanes 0-15 sits in lane l + 16. The loads that do not
// depend on the row's sequence (split partials, gamma) are issued first; the
// sequence is found with one ballot over cu_rows, so the dependent chain is
// cu_rows -> lens -> RoPE row.
__device__ __forceinline__ void head_row_bf16(const HeadEpilogue& e, int wid, int lane) {
  const int heads = e.n_q + 2 * e.n_kv;
  if (wid >= e.rows * heads) return;
  const int row = wid / heads, head = wid - row * heads;
  const int kind = head < e.n_q ? 0 : (head < e.n_q + e.n_kv ? 1 : 2);  // Q, K, V
  // split-K partials of this (row, head): eight splits per round trip, added in pairs
  const size_t split_stride4 = (size_t)e.rows * e.ldY / 4;
  const float4* y4 = reinterpret_cast<const float4*>(e.Y + (size_t)row * e.ldY + (size_t)head * 128) + lane;
  float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < e.splits; s0 += 8) {
    float4 a[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      a[j] = s0 + j < e.splits ? y4[(s0 + j) * split_stride4] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      x.x += a[j].x + a[j + 1].x;
      x.y += a[j].y + a[j + 1].y;
      x.z += a[j].z + a[j + 1].z;
      x.w += a[j].w + a[j + 1].w;
    }
  }
  float4 g = make_float4(1.f, 1.f, 1.f, 1.f);
  if (kind < 2) {  // gamma has no alignment guarantee beyond its element size
    const bf16* gp = (const bf16*)(kind == 0 ? e.gamma_q : e.gamma_k) + 4 * lane;
    g = make_float4(__bfloat162float(gp[0]), __bfloat162float(gp[1]), __bfloat162float(gp[2]),
                    __bfloat162float(gp[3]));
  }
  int b, t, n_b;
  if (e.cu_rows) {
    // b = number of sequences 1..batch-1 that start at or before this row
    b = 0;
    for (int base = 1; base < e.batch; base += 32) {
      const int j = base + lane;
      b += __popc(__ballot_sync(0xffffffffu, j < e.batch && e.cu_rows[j] <= row));
    }
    const int r0 = e.cu_rows[b], r1 = e.cu_rows[b + 1];
    t = row - r0;
    n_b = r1 - r0;
    if (n_b < 0 || r1 > e.rows || e.cu_rows[0] != 0 || t < 0 || t >= n_b) {
      if (lane == 0) atomicOr(e.status, DFLASH_DEV_ROWS);
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
    if (lane == 0 && t == 0 && head == 0)
      atomicOr(e.status, (start + n_b > e.capacity || start < 0) ? DFLASH_DEV_CAPACITY
                                                                 : DFLASH_DEV_ROPE);
    return;
  }
  const int pos = start + t;
  if (kind < 2) {
    const float2* cs = e.rope + (size_t)pos * 64 + 4 * (lane & 15);  // (cos, sin), dims 4l.. mod 64
    const float2 c0 = cs[0], c1 = cs[1], c2 = cs[2], c3 = cs[3];
    const float ss = warp_sum(x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w);
    const float r = 1.0f / sqrtf(ss * (1.0f / 128.f) + e.eps);
    x.x *= r * g.x;
    x.y *= r * g.y;
    x.z *= r * g.z;
    x.w *= r * g.w;
    // partner values: dims i + 64 for lanes 0-15, i - 64 for lanes 16-31
    float4 o;
    o.x = __shfl_xor_sync(0xffffffffu, x.x, 16);
    o.y = __shfl_xor_sync(0xffffffffu, x.y, 16);
    o.z = __shfl_xor_sync(0xffffffffu, x.z, 16);
    o.w = __shfl_xor_sync(0xffffffffu, x.w, 16);
    const float sg = lane < 16 ? -1.f : 1.f;  // rotate_half: [-x2; x1]
    x.x = x.x * c0.x + sg * o.x * c0.y;
    x.y = x.y * c1.x + sg * o.y * c1.y;
    x.z = x.z * c2.x + sg * o.z * c2.y;
    x.w = x.w * c3.x + sg * o.w * c3.y;
  }
  // element offset of the destination row: Q, or the cache slot
  size_t eoff;
  if (kind == 0) {
    eoff = (((size_t)b * e.n_q + head) * e.bs + t) * 128;
  } else {
    const int kvh = head - e.n_q - (kind == 2 ? e.n_kv : 0);
    eoff = cache_row(e.block_table, e.pages_per_seq, e.n_kv, e.capacity, b, kvh, pos) * 128;
  }
  char* base = (char*)(kind == 0 ? e.q_out : kind == 1 ? e.cache_k : e.cache_v);
  if (e.kv_fp8) {
    // E4M3: Q as codes + remainder codes, K / V as codes of x / scale
    if (kind == 0) {
      uint32_t hi, lo;
      e4m3x4_split(x.x, x.y, x.z, x.w, hi, lo);
      reinterpret_cast<uint32_t*>(base + eoff)[lane] = hi;
      reinterpret_cast<uint32_t*>((char*)e.q_lo + eoff)[lane] = lo;
    } else {
      const float inv = kind == 1 ? e.k_inv : e.v_inv;
      reinterpret_cast<uint32_t*>(base + eoff)[lane] =
          e4m3x4(x.x * inv, x.y * inv, x.z * inv, x.w * inv);
    }
    return;
  }
  bf16* dst = (bf16*)base + eoff;
  __nv_bfloat162 lo2 = __floats2bfloat162_rn(x.x, x.y), hi2 = __floats2bfloat162_rn(x.z, x.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&lo2);
  u.y = *reinterpret_cast<uint32_t*>(&hi2);
  reinterpret_cast<uint2*>(dst)[lane] = u;
}

__global__ void __launch_bounds__(256) head_epilogue_bf16_kernel(const __grid_constant__ HeadEpilogue e) {
  head_row_bf16(e, blockIdx.x * 8 + (threadIdx.x >> 5), threadIdx.x & 31);
}

// Two epilogues in one launch (an inject's context rows and the block's rows of the same
// layer): warps [0, w0) finish e0's (row, head) pairs, the rest e1's.
__global__ void __launch_bounds__(256) head_epilogue_bf16_pair_kernel(
    const __grid_constant__ HeadEpilogue e0, const __grid_constant__ HeadEpilogue e1, int w0) {
  const int wid = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (wid < w0)
    head_row_bf16(e0, wid, threadIdx.x & 31);
  else
    head_row_bf16(e1, wid - w0, threadIdx.x & 31);
}

__global__ void lens_advance_kernel(int32_t* lens, const int32_t* cu_rows, int batch, int bs,
                                    int M, int capacity, int table_len) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= batch) return;
  int n_b = bs;
  if (cu_rows) {
    n_b = cu_rows[b + 1] - cu_rows[b];
    if (n_b < 0 || cu_rows[b + 1] > M || cu_rows[0] != 0) return;
  }
  const int start = lens[b];
  if (start < 0 || start + n_b > capacity || start + n_b > table_len) return;
  lens[b] = start + n_b;
}

__global__ void crop_kernel(int32_t* lens, int n_layers, int batch, const int32_t* new_lens,
                            unsigned* status) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_layers * batch) return;
  const int b = i % batch;
  const int n = new_lens[b];
  if (n < 0 || n > lens[i]) {
    atomicOr(status, DFLASH_DEV_CROP);
    return;
  }
  lens[i] = n;
}

__global__ void rope_table_kernel(double theta, int d_h, int max_pos, float2* table) {
  const int half = d_h / 2;
  const size_t n = (size_t)max_pos * half;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < n;
       e += (size_t)gridDim.x * blockDim.x) {
    const int p = (int)(e / half), i = (int)(e % half);
    const double w = pow(theta, -2.0 * (double)i / (double)d_h);
    double sn, cs;
    sincos((double)p * w, &sn, &cs);
    table[e] = make_float2((float)cs, (float)sn);
  }
}

// smallest per-thread chunk count (1, 2, 4 or 8 float4) that covers the row; with few rows
// (fewer than 64) a CTA of 1024 threads per row, whose threads then hold one or two chunks
// and load eight splits at a time
template <typename T>
void launch_norm(int M, cudaStream_t s, const float* Y, int splits, int N, const T* gamma,
                 float eps, T* out) {
  if (M < 64 && N / 4 <= 2 * 1024) {
    if (N / 4 <= 1024)
      rmsnorm_rows_vec_kernel<T, 1, 1024><<<M, 1024, 0, s>>>(Y, splits, M, N, gamma, eps, out);
    else
      rmsnorm_rows_vec_kernel<T, 2, 1024><<<M, 1024, 0, s>>>(Y, splits, M, N, gamma, eps, out);
    return;
  }
  const int need = (N / 4 + kNormThreads - 1) / kNormThreads;
  if (need <= 1)
    rmsnorm_rows_vec_kernel<T, 1, kNormThreads><<<M, kNormThreads, 0, s>>>(Y, splits, M, N, gamma, eps, out);
  else if (need <= 2)
    rmsnorm_rows_vec_kernel<T, 2, kNormThreads><<<M, kNormThreads, 0, s>>>(Y, splits, M, N, gamma, eps, out);
  else if (need <= 4)
    rmsnorm_rows_vec_kernel<T, 4, kNormThreads><<<M, kNormThreads, 0, s>>>(Y, splits, M, N, gamma, eps, out);
  else
    rmsnorm_rows_vec_kernel<T, 8, kNormThreads><<<M, kNormThreads, 0, s>>>(Y, splits, M, N, gamma, eps, out);
}

}  // namespace

cudaError_t rmsnorm_rows(int dtype, const float* Y, int splits, int M, int N, const void* gamma,
                         float eps, void* out, cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  // the vector kernel loads gamma 4 elements at a time (8-byte aligned for bf16)
  if (N % 4 == 0 && N <= 4 * kNormThreads * kNormMaxChunks &&
      (dtype == DFLASH_F32 || ((uintptr_t)gamma & 7) == 0)) {
    LaunchScope ls_(DFLASH_KERNEL_RMSNORM, s);
    if (dtype == DFLASH_F32)
      launch_norm<float>(M, s, Y, splits, N, (const float*)gamma, eps, (float*)out);
    else
      launch_norm<bf16>(M, s, Y, splits, N, (const bf16*)gamma, eps, (bf16*)out);
    return cudaGetLastError();
  }
  if (dtype == DFLASH_F32)
    {
      LaunchScope ls_(DFLASH_KERNEL_RMSNORM, s);
      rmsnorm_rows_kernel<float><<<M, 256, 0, s>>>(Y, splits, M, N, (const float*)gamma, eps,
                                                   (float*)out);
    }
  else
    {
      LaunchScope ls_(DFLASH_KERNEL_RMSNORM, s);
      rmsnorm_rows_kernel<bf16><<<M, 256, 0, s>>>(Y, splits, M, N, (const bf16*)gamma, eps,
                                                  (bf16*)out);
    }
  return cudaGetLastError();
}

cudaError_t head_epilogue(int dtype, const HeadEpilogue& e, cudaStream_t s) {
  if (e.rows <= 0) return cudaSuccess;
  dim3 grid(e.n_q + 2 * e.n_kv, e.rows);
  int threads = ((e.d_h / 2 + 31) / 32) * 32;
  if (dtype == DFLASH_F32)
    {
      LaunchScope ls_(DFLASH_KERNEL_HEAD_EPILOGUE, s);
      head_epilogue_kernel<float><<<grid, threads, 0, s>>>(e);
    }
  else
    {
      LaunchScope ls_(DFLASH_KERNEL_HEAD_EPILOGUE, s);
      head_epilogue_kernel<bf16><<<grid, threads, 0, s>>>(e);
    }
  return cudaGetLastError();
}

cudaError_t head_epilogue_bf16(const HeadEpilogue& e, cudaStream_t s) {
  if (e.rows <= 0) return cudaSuccess;
  if (e.d_h != 128) return cudaErrorInvalidValue;
  const long long warps = (long long)e.rows * (e.n_q + 2 * e.n_kv);
  {
    LaunchScope ls_(DFLASH_KERNEL_HEAD_EPILOGUE, s);
    head_epilogue_bf16_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, s>>>(e);
  }
  return cudaGetLastError();
}

cudaError_t head_epilogue_bf16_pair(const HeadEpilogue& e0, const HeadEpilogue& e1,
                                    cudaStream_t s) {
  if (e0.d_h != 128 || e1.d_h != 128) return cudaErrorInvalidValue;
  const long long w0 = e0.rows > 0 ? (long long)e0.rows * (e0.n_q + 2 * e0.n_kv) : 0;
  const long long w1 = e1.rows > 0 ? (long long)e1.rows * (e1.n_q + 2 * e1.n_kv) : 0;
  if (w0 + w1 == 0) return cudaSuccess;
  if (w0 + w1 >= (1ll << 31) - 8) return cudaErrorInvalidValue;
  {
    LaunchScope ls_(DFLASH_KERNEL_HEAD_EPILOGUE, s);
    head_epilogue_bf16_pair_kernel<<<(unsigned)((w0 + w1 + 7) / 8), 256, 0, s>>>(e0, e1, (int)w0);
  }
  return cudaGetLastError();
}

cudaError_t lens_advance(int32_t* lens, const int32_t* cu_rows, int batch, int bs, int M,
                         int capacity, int table_len, cudaStream_t s) {
  {
    LaunchScope ls_(DFLASH_KERNEL_LENS, s);
    lens_advance_kernel<<<(batch + 127) / 128, 128, 0, s>>>(lens, cu_rows, batch, bs, M, capacity,
                                                            table_len);
  }
  return cudaGetLastError();
}

cudaError_t crop_lens(int32_t* lens, int n_layers, int batch, const int32_t* new_lens,
                      unsigned* status, cudaStream_t s) {
  const int n = n_layers * batch;
  {
    LaunchScope ls_(DFLASH_KERNEL_CROP, s);
    crop_kernel<<<(n + 127) / 128, 128, 0, s>>>(lens, n_layers, batch, new_lens, status);
  }
  return cudaGetLastError();
}

cudaError_t rope_table(double theta, int d_h, int max_pos, float* table, cudaStream_t s) {
  const size_t n = (size_t)max_pos * (d_h / 2);
  int blocks = (int)((n + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  {
    LaunchScope ls_(DFLASH_KERNEL_ROPE_TABLE, s);
    rope_table_kernel<<<blocks, 256, 0, s>>>(theta, d_h, max_pos, (float2*)table);
  }
  return cudaGetLastError();
}

}  // namespace dflash
