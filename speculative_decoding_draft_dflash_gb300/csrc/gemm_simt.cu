// SIMT GEMM with fp32 accumulation: Y[M][N] = X[M][K] W[N][K]^T.
//
// The fp32 path of the library (the walkthrough-sized single layer) runs its
// projections here: FFMA keeps full fp32 products, where a TF32 tensor-core
// product would lose about 11 bits per term. X arrives as up to eight
// K-segments (the k target layers' hidden states, never concatenated).
#include "dflash_internal.cuh"

namespace dflash {
namespace {

constexpr int BM = 64, BN = 64, BK = 16, NT = 256;

template <typename T>
__global__ void __launch_bounds__(NT) gemm_simt_kernel(Segments A, int M, Weights W, float* Y,
                                                       int ldY) {
  const int N = W.total();
  __shared__ float As[BK][BM + 4];
  __shared__ float Ws[BK][BN + 4];
  const int K = A.n * A.kseg;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += BK) {
    // 64 x 16 elements of each operand, 4 per thread
    for (int e = threadIdx.x; e < BM * BK; e += NT) {
      int r = e / BK, c = e % BK;
      int gm = m0 + r, gk = k0 + c;
      float a = 0.f;
      if (gm < M && gk < K) {
        int seg = gk / A.kseg, kk = gk - seg * A.kseg;
        a = to_f(((const T*)A.p[seg])[(size_t)gm * A.kseg + kk]);
      }
      As[c][r] = a;
      int gn = n0 + r;
      float wv = 0.f;
      if (gn < N && gk < K) {
        int wi = 0, off = 0;
        while (wi + 1 < W.count && gn >= off + W.n[wi]) off += W.n[wi++];
        wv = to_f(((const T*)W.p[wi])[(size_t)(gn - off) * K + gk]);
      }
      Ws[c][r] = wv;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Ws[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int gm = m0 + ty * 4 + i;
    if (gm >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int gn = n0 + tx * 4 + j;
      if (gn < N) Y[(size_t)gm * ldY + gn] = acc[i][j];
    }
  }
}

}  // namespace

cudaError_t gemm_simt(int dtype, const Segments& A, int M, const Weights& W, float* Y, int ldY,
                      cudaStream_t s) {
  const int N = W.total();
  if (M <= 0 || N <= 0) return cudaSuccess;
  dim3 grid((N + BN - 1) / BN, (M + BM - 1) / BM);
  if (dtype == DFLASH_F32)
    {
      LaunchScope ls_(DFLASH_KERNEL_GEMM, s);
      gemm_simt_kernel<float><<<grid, NT, 0, s>>>(A, M, W, Y, ldY);
    }
  else
    {
      LaunchScope ls_(DFLASH_KERNEL_GEMM, s);
      gemm_simt_kernel<bf16><<<grid, NT, 0, s>>>(A, M, W, Y, ldY);
    }
  return cudaGetLastError();
}

}  // namespace dflash
