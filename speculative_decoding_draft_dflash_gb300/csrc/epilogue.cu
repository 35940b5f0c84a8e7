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
#include "dflash_internal.cuh"

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
  const int start = e.lens[b];
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
    dst = base + (((size_t)b * e.n_kv + kvh) * e.capacity + pos) * e.d_h;
  }
  dst[i] = from_f<T>(x0);
  dst[i + half] = from_f<T>(x1);
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

}  // namespace

cudaError_t rmsnorm_rows(int dtype, const float* Y, int splits, int M, int N, const void* gamma,
                         float eps, void* out, cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
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
