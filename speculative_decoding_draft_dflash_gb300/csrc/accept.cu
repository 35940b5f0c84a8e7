// Acceptance bookkeeping of a verified round, on the device (DFlash KV Injection
// Walkthrough, Step 6: accepted length = leading matches of the block's tokens 1..bs-1
// against the target's posterior tokens 0..bs-2; Step 7: start += a + 1, the next round
// injects the a + 1 context rows of the anchor and the accepted tokens, and the target's
// token after the accepted prefix is the next block's anchor). The next inject's row
// offsets are a prefix sum over the sequences, so the whole round state stays on the
// device and the host never reads an acceptance length.
#include "dflash_internal.cuh"

namespace dflash {
namespace {

// One CTA: per sequence the accepted length (bs <= a few dozen comparisons), then a
// CTA-wide inclusive scan of the next inject counts, chunk by chunk with a carry.
__global__ void __launch_bounds__(1024) accept_kernel(const int32_t* __restrict__ block_ids,
                                                      const int32_t* __restrict__ posterior,
                                                      int batch, int bs,
                                                      const int32_t* __restrict__ ctx_len,
                                                      int32_t* accept_len, int32_t* cu,
                                                      int32_t* ctx_next, int32_t* anchor) {
  __shared__ int warp_tot[32];
  __shared__ int carry;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if (threadIdx.x == 0) {
    carry = 0;
    cu[0] = 0;
  }
  __syncthreads();
  for (int base = 0; base < batch; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int cnt = 0;
    if (b < batch) {
      const int32_t* blk = block_ids + (size_t)b * bs;
      const int32_t* post = posterior + (size_t)b * bs;
      int a = 0;
      while (a < bs - 1 && blk[a + 1] == post[a]) ++a;
      accept_len[b] = a;
      anchor[b] = post[a];
      ctx_next[b] = ctx_len[b] + a + 1;
      cnt = a + 1;
    }
    // inclusive scan: within the warp, then over the warp totals
    int v = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += u;
    }
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    if (warp == 0) {
      int t = lane < nw ? warp_tot[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, t, o);
        if (lane >= o) t += u;
      }
      if (lane < nw) warp_tot[lane] = t;  // inclusive totals up to each warp
    }
    __syncthreads();
    const int before = carry + (warp > 0 ? warp_tot[warp - 1] : 0);
    if (b < batch) cu[b + 1] = before + v;
    __syncthreads();
    if (threadIdx.x == 0) carry += warp_tot[nw - 1];
    __syncthreads();
  }
}

}  // namespace

cudaError_t accept_round(const int32_t* block_ids, const int32_t* posterior, int batch, int bs,
                         const int32_t* ctx_len, int32_t* accept_len, int32_t* cu,
                         int32_t* ctx_next, int32_t* anchor, cudaStream_t s) {
  LaunchScope ls_(DFLASH_KERNEL_ACCEPT, s);
  accept_kernel<<<1, 1024, 0, s>>>(block_ids, posterior, batch, bs, ctx_len, accept_len, cu,
                                   ctx_next, anchor);
  return cudaGetLastError();
}

}  // namespace dflash
