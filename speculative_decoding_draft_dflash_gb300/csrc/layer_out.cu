// The rest of a draft decoder layer after its attention (DFlash KV Injection
// Walkthrough, Step 4.5: the concatenated heads times W_O; Step 5: the draft's decoder
// layers, read as Qwen3 pre-norm residual layers with a SwiGLU MLP):
//
//   x1  = x + attn_out W_O^T                 o_proj GEMM, then rows_kernel (residual,
//   n   = RMSNorm_post(x1)                   split-K sum and the norm in one pass)
//   h   = silu(n W_gate^T) * (n W_up^T)      one GEMM over the stacked [W_gate | W_up],
//                                            then swiglu_kernel
//   out = x1 + h W_down^T                    down GEMM, then rows_kernel (residual)
//
// The GEMMs are the library's projection GEMMs (tcgen05 for bf16, FFMA for fp32) with
// fp32 split-K partials; the row kernels are HBM-bound and vectorised by four columns.
#include "dflash_internal.cuh"

namespace dflash {
namespace {

constexpr int kRowThreads = 256, kRowMaxChunks = 8;

template <typename T>
__device__ __forceinline__ float4 load4(const T* p);
template <>
__device__ __forceinline__ float4 load4<float>(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}
template <>
__device__ __forceinline__ float4 load4<bf16>(const bf16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

template <typename T>
__device__ __forceinline__ void store4(T* p, float4 v);
template <>
__device__ __forceinline__ void store4<float>(float* p, float4 v) {
  *reinterpret_cast<float4*>(p) = v;
}
template <>
__device__ __forceinline__ void store4<bf16>(bf16* p, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

__device__ __forceinline__ float cta_sum(float v, float* red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31, nw = blockDim.x >> 5;
  if (l == 0) red[w] = v;
  __syncthreads();
  float t = 0.f;
  for (int i = 0; i < nw; ++i) t += red[i];
  __syncthreads();
  return t;
}

// One CTA per row: v = resid + sum of `splits` fp32 partials (either may be absent);
// stores v to sum_out and RMSNorm(v) * gamma to norm_out (either may be absent).
template <typename T, int CH>
__global__ void __launch_bounds__(kRowThreads) rows_kernel(const float* __restrict__ Y, int splits,
                                                           const T* __restrict__ resid,
                                                           T* __restrict__ sum_out,
                                                           const T* __restrict__ gamma, float eps,
                                                           T* __restrict__ norm_out, int M, int N) {
  __shared__ float red[32];
  const int row = blockIdx.x;
  const int n4 = N >> 2;
  const size_t split_stride = (size_t)M * N;
  float4 v[CH];
#pragma unroll
  for (int k = 0; k < CH; ++k) {
    const int c = threadIdx.x + k * kRowThreads;
    v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c < n4 && resid) v[k] = load4(resid + (size_t)row * N + 4 * c);
  }
  for (int s = 0; s < splits; ++s) {
    float4 a[CH];
#pragma unroll
    for (int k = 0; k < CH; ++k) {
      const int c = threadIdx.x + k * kRowThreads;
      a[k] = c < n4 ? load4(Y + s * split_stride + (size_t)row * N + 4 * c) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < CH; ++k) {
      v[k].x += a[k].x;
      v[k].y += a[k].y;
      v[k].z += a[k].z;
      v[k].w += a[k].w;
    }
  }
  if (sum_out) {
#pragma unroll
    for (int k = 0; k < CH; ++k) {
      const int c = threadIdx.x + k * kRowThreads;
      if (c < n4) store4<T>(sum_out + (size_t)row * N + 4 * c, v[k]);
    }
  }
  if (!norm_out) return;
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < CH; ++k)
    ss += v[k].x * v[k].x + v[k].y * v[k].y + v[k].z * v[k].z + v[k].w * v[k].w;
  ss = cta_sum(ss, red);
  const float r = 1.0f / sqrtf(ss / (float)N + eps);
#pragma unroll
  for (int k = 0; k < CH; ++k) {
    const int c = threadIdx.x + k * kRowThreads;
    if (c < n4) {
      const float4 g = load4(gamma + 4 * c);
      store4<T>(norm_out + (size_t)row * N + 4 * c,
                make_float4(v[k].x * r * g.x, v[k].y * r * g.y, v[k].z * r * g.z, v[k].w * r * g.w));
    }
  }
}

// h[m][j] = silu(g) * u, g and u summed over the split-K partials of the stacked
// projection Y[s][m][0 .. 2F): gate columns first, then up columns.
template <typename T>
__global__ void swiglu_kernel(const float* __restrict__ Y, int splits, int M, int F,
                              T* __restrict__ h) {
  const size_t n4 = (size_t)M * F / 4;
  const size_t split_stride = (size_t)M * 2 * F;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t e = 4 * i, m = e / F, j = e - m * F;
    float4 g = make_float4(0.f, 0.f, 0.f, 0.f), u = g;
    for (int s = 0; s < splits; ++s) {
      const float* y = Y + s * split_stride + m * 2 * F;
      const float4 a = *reinterpret_cast<const float4*>(y + j);
      const float4 b = *reinterpret_cast<const float4*>(y + F + j);
      g.x += a.x; g.y += a.y; g.z += a.z; g.w += a.w;
      u.x += b.x; u.y += b.y; u.z += b.z; u.w += b.w;
    }
    auto silu = [](float x) { return x / (1.0f + __expf(-x)); };
    store4<T>(h + m * F + j, make_float4(silu(g.x) * u.x, silu(g.y) * u.y, silu(g.z) * u.z,
                                         silu(g.w) * u.w));
  }
}

template <typename T>
cudaError_t launch_rows(int M, int N, const float* Y, int splits, const T* resid, T* sum_out,
                        const T* gamma, float eps, T* norm_out, cudaStream_t s) {
  const int need = (N / 4 + kRowThreads - 1) / kRowThreads;
  LaunchScope ls_(DFLASH_KERNEL_RMSNORM, s);
  if (need <= 1)
    rows_kernel<T, 1><<<M, kRowThreads, 0, s>>>(Y, splits, resid, sum_out, gamma, eps, norm_out, M, N);
  else if (need <= 2)
    rows_kernel<T, 2><<<M, kRowThreads, 0, s>>>(Y, splits, resid, sum_out, gamma, eps, norm_out, M, N);
  else if (need <= 4)
    rows_kernel<T, 4><<<M, kRowThreads, 0, s>>>(Y, splits, resid, sum_out, gamma, eps, norm_out, M, N);
  else
    rows_kernel<T, 8><<<M, kRowThreads, 0, s>>>(Y, splits, resid, sum_out, gamma, eps, norm_out, M, N);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_swiglu(const float* Y, int splits, int M, int F, T* h, cudaStream_t s) {
  const size_t n4 = (size_t)M * F / 4;
  const int blocks = (int)((n4 + 255) / 256 < 4096 ? (n4 + 255) / 256 : 4096);
  LaunchScope ls_(DFLASH_KERNEL_HEAD_EPILOGUE, s);
  swiglu_kernel<T><<<blocks > 0 ? blocks : 1, 256, 0, s>>>(Y, splits, M, F, h);
  return cudaGetLastError();
}

Segments one_segment(const void* X, int K) {
  Segments A;
  A.n = 1;
  A.kseg = K;
  A.p[0] = X;
  return A;
}

Weights one_weight(const void* W, int N) {
  Weights w;
  w.p[0] = W;
  w.n[0] = N;
  w.count = 1;
  return w;
}

}  // namespace

bool rows_ok(int N) { return N % 4 == 0 && N <= 4 * kRowThreads * kRowMaxChunks; }

cudaError_t norm_rows(int dtype, int M, int N, const void* x, const void* gamma, float eps,
                      void* out, cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  if (dtype == DFLASH_F32)
    return launch_rows<float>(M, N, nullptr, 0, (const float*)x, nullptr, (const float*)gamma,
                              eps, (float*)out, s);
  return launch_rows<bf16>(M, N, nullptr, 0, (const bf16*)x, nullptr, (const bf16*)gamma, eps,
                           (bf16*)out, s);
}

LayerOutScratch carve_layer_out(Carver& cv, int dtype, int M, int d, int a_dim, int d_ff) {
  LayerOutScratch sc;
  sc.splits_o = gemm_splits(dtype, M, one_weight(nullptr, d), a_dim);
  Weights gu;
  gu.p[0] = gu.p[1] = nullptr;
  gu.n[0] = gu.n[1] = d_ff;
  gu.count = 2;
  sc.splits_gu = gemm_splits(dtype, M, gu, d);
  sc.splits_d = gemm_splits(dtype, M, one_weight(nullptr, d), d_ff);
  const int so = sc.splits_o > sc.splits_d ? sc.splits_o : sc.splits_d;
  const size_t es = dtype == DFLASH_F32 ? 4 : 2;
  sc.Y = cv.take<float>((size_t)so * M * d);
  sc.Ygu = cv.take<float>((size_t)sc.splits_gu * M * 2 * d_ff);
  sc.x1 = cv.take<char>((size_t)M * d * es);
  sc.n = cv.take<char>((size_t)M * d * es);
  sc.h = cv.take<char>((size_t)M * d_ff * es);
  return sc;
}

cudaError_t layer_out(int dtype, int M, int d, int a_dim, int d_ff, const void* attn_out,
                      const void* x, const void* W_O, const void* gamma_post, float eps,
                      const void* W_gate, const void* W_up, const void* W_down, void* x_out,
                      const LayerOutScratch& sc, unsigned* status, cudaStream_t s) {
  const bool f32 = dtype == DFLASH_F32;
  // x1 = x + attn_out W_O^T and n = RMSNorm_post(x1)
  cudaError_t e = gemm(dtype, one_segment(attn_out, a_dim), M, one_weight(W_O, d), sc.Y, d, status, s);
  if (e != cudaSuccess) return e;
  e = f32 ? launch_rows<float>(M, d, sc.Y, sc.splits_o, (const float*)x, (float*)sc.x1,
                               (const float*)gamma_post, eps, (float*)sc.n, s)
          : launch_rows<bf16>(M, d, sc.Y, sc.splits_o, (const bf16*)x, (bf16*)sc.x1,
                              (const bf16*)gamma_post, eps, (bf16*)sc.n, s);
  if (e != cudaSuccess) return e;
  // h = silu(n W_gate^T) * (n W_up^T)
  Weights gu;
  gu.p[0] = W_gate;
  gu.p[1] = W_up;
  gu.n[0] = gu.n[1] = d_ff;
  gu.count = 2;
  e = gemm(dtype, one_segment(sc.n, d), M, gu, sc.Ygu, 2 * d_ff, status, s);
  if (e != cudaSuccess) return e;
  e = f32 ? launch_swiglu<float>(sc.Ygu, sc.splits_gu, M, d_ff, (float*)sc.h, s)
          : launch_swiglu<bf16>(sc.Ygu, sc.splits_gu, M, d_ff, (bf16*)sc.h, s);
  if (e != cudaSuccess) return e;
  // out = x1 + h W_down^T
  e = gemm(dtype, one_segment(sc.h, d_ff), M, one_weight(W_down, d), sc.Y, d, status, s);
  if (e != cudaSuccess) return e;
  return f32 ? launch_rows<float>(M, d, sc.Y, sc.splits_d, (const float*)sc.x1, (float*)x_out,
                                  nullptr, 0.f, nullptr, s)
             : launch_rows<bf16>(M, d, sc.Y, sc.splits_d, (const bf16*)sc.x1, (bf16*)x_out,
                                 nullptr, 0.f, nullptr, s);
}

}  // namespace dflash
