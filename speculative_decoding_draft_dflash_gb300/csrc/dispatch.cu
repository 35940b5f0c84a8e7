// Per-dtype choice of GEMM and attention kernels.
#include "dflash_internal.cuh"

namespace dflash {

int gemm_splits(int dtype, int M, const Weights& W, int K, int split_cap) {
  return dtype == DFLASH_F32 ? 1 : gemm_tc_splits(M, W, K, split_cap);
}

cudaError_t gemm(int dtype, const Segments& A, int M, const Weights& W, float* Y, int ldY,
                 unsigned* status, cudaStream_t s, int split_cap) {
  if (dtype == DFLASH_F32) return gemm_simt(dtype, A, M, W, Y, ldY, s);
  return gemm_tc(A, M, W, Y, ldY, status, s, split_cap);
}

int attn_chunk(int dtype) { return dtype == DFLASH_F32 ? attn_simt_chunk() : attn_tc_chunk(); }

cudaError_t attention(int dtype, const AttnParams& p, cudaStream_t s) {
  return dtype == DFLASH_F32 ? attn_simt(dtype, p, s) : attn_tc(p, s);
}

}  // namespace dflash
