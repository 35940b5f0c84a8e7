// Work list of the tensor-core block attention, computed by one CTA.
//
// For every sequence b the block occupies positions start .. start + bs - 1,
// start = lens[b] plus the rows a KV inject issued in the same call appended
// (DFlash KV Injection Walkthrough, Step 7: the cache grows by the new context
// rows, then the block follows them). The keys a query of the block sees are
// [lo, start + bs): the whole prefix, or the last W positions under a sliding
// window of W (the window reading of the hybrid layers).
//
// A CTA's time is close to a fixed cost per 128-key tile plus a fixed cost per item
// (the last tile's V load, the output stores, the next item's first S), so the work is
// split by that cost: the key ranges of all (sequence, KV head) pairs, laid end to end in
// pair order, each as an item header followed by its tiles, form one cost stream of
// total W, and CTA c of n takes the tiles whose centres fall in [c W / n, (c + 1) W / n).
// A range that straddles a boundary becomes several items (split ranges, merged
// afterwards by the combine kernel). CTAs whose shares hold many short ranges then get
// fewer tiles, and all finish at about the same time.
//
// The same pass records, per sequence, the block start (read by the attention
// for the window test) and the cache length after the call, which the combine
// kernel writes back once the attention has finished with the old lengths.
#pragma once

#include <climits>

#include "dflash_internal.cuh"

namespace dflash {
namespace sched {

constexpr int kTileKeys = 128;     // keys per attention tile
// a key range is cut into at most ceil(keys / (kItemMinTiles * kTileKeys)) items (the
// partial rows kept per (sequence, KV head) pair)
constexpr int kItemMinTiles = 4;
constexpr int kShareMinTiles = 2;  // smallest share of a CTA worth its pipeline ramp
constexpr int kTileCost = 8;       // cost of a tile in the partition (even: tile centres)
constexpr int kMaxSm = 256;        // most CTAs a list is built for
constexpr int kMergeCountShift = 20;  // merge_list entry: pair | item count << this

struct Params {
  const int32_t* lens;      // [batch] lengths before the call
  const int32_t* pre_rows;  // cu_rows [batch + 1] of rows injected in the same call, or null
  int pre_M;                // row count of that inject
  int4* items;              // [n_sm]: the item each CTA takes first (the last of its share),
                            // then [n_sm + i]: item i of the list; an item is
                            // {pair, k_begin, k_end, split (-1 = whole range)}
  int* first;               // [n_sm + 1]: CTA c takes list items first[c] .. first[c + 1] - 1
  int* n_items;             // list length
  int* splits;              // [pair]: items of the pair (0 = refused sequence)
  int* merge_list;          // pairs whose rows the combine writes (split or refused), each
  int* n_merge;             //   with its item count (pair | n << kMergeCountShift); how many
  int* ready;               // set to 1 once the list is complete (the attention clears it)
  int32_t* qstart;          // [batch]: first position of the block
  int32_t* lens_new;        // [batch]: length after the call
  int batch, n_kv, bs, window, capacity, table_len, max_splits, n_sm;
  int align;                // key ranges start on multiples of this (paged cache: a page)
  int item_cost;            // cost of an item's header, on the scale of kTileCost per tile
};

// Bytes of the work-list area for `pairs` (sequence, KV head) pairs of `batch` sequences
// on n_sm CTAs: items (2 n_sm + pairs), first (n_sm + 1), splits, 16 counters, qstart,
// lens_new, merge_list. The list has at most pairs + n_sm - 1 items (each CTA boundary
// cuts at most one range).
inline size_t area_bytes(size_t pairs, size_t batch, size_t n_sm) {
  return (2 * n_sm + pairs) * 16 + (n_sm + 1) * 4 + pairs * 4 + 64 + batch * 8 + pairs * 4;
}

// Rows the inject of the same call appended for sequence b: all of its rows when they
// fit the cache and the RoPE table (the condition under which the inject advances the
// length), else none.
__device__ __forceinline__ int injected_rows(const int32_t* cu_rows, int M, int b, int start,
                                             int capacity, int table_len) {
  if (!cu_rows) return 0;
  const int r0 = cu_rows[b], r1 = cu_rows[b + 1];
  const int n = r1 - r0;
  if (n < 0 || r1 > M || cu_rows[0] != 0) return 0;
  if (start < 0 || start + n > capacity || start + n > table_len) return 0;
  return n;
}

struct Range {
  int start, end, lo;
  bool ok;  // the block fits the cache and the RoPE table
};

__device__ __forceinline__ Range seq_range(const Params& p, int b) {
  Range r;
  const int l = p.lens[b];
  r.start = l + injected_rows(p.pre_rows, p.pre_M, b, l, p.capacity, p.table_len);
  r.end = r.start + p.bs;
  r.lo = p.window > 0 ? max(0, r.start - p.window + 1) : 0;
  r.lo -= r.lo % p.align;  // keys below the window's start are masked by the window test
  r.ok = r.start >= 0 && r.end <= p.capacity && r.end <= p.table_len;
  return r;
}

// Exclusive prefix sum of v over the CTA's threads in thread order; *total receives the
// sum. tmp: 32 ints of shared memory.
__device__ __forceinline__ int cta_scan(int v, int* tmp, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = (int)(blockDim.x >> 5);
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tmp[w] = x;
  __syncthreads();
  int base = 0, tot = 0;
  for (int i = 0; i < nw; ++i) {
    base += i < w ? tmp[i] : 0;
    tot += tmp[i];
  }
  __syncthreads();
  *total = tot;
  return base + x - v;
}

__device__ __forceinline__ int cta_max(int v, int* tmp) {
  v = __reduce_max_sync(0xffffffffu, v);
  if ((threadIdx.x & 31) == 0) tmp[threadIdx.x >> 5] = v;
  __syncthreads();
  int m = 0;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) m = max(m, tmp[i]);
  __syncthreads();
  return m;
}

// Minimum of v over threads threadIdx.x .. blockDim.x - 1 (a suffix minimum in thread
// order). tmp: 32 ints of shared memory.
__device__ __forceinline__ int cta_suffix_min(int v, int* tmp) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = (int)(blockDim.x >> 5);
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_down_sync(0xffffffffu, x, o);
    if (lane + o < 32) x = min(x, y);
  }
  if (lane == 0) tmp[w] = x;
  __syncthreads();
  for (int i = w + 1; i < nw; ++i) x = min(x, tmp[i]);
  __syncthreads();
  return x;
}

// Tiles of pair pr's key range (0 for a refused sequence).
__device__ __forceinline__ int pair_tiles(const Params& p, int pr) {
  const Range r = seq_range(p, pr / p.n_kv);
  return r.ok ? (r.end - r.lo + kTileKeys - 1) / kTileKeys : 0;
}

// Run by every thread of one CTA (blockDim.x a multiple of 32, n_sm <= kMaxSm).
inline __device__ void build(const Params& p) {
  __shared__ int tmp[32];
  __shared__ int s_merge;
  __shared__ int s_first[kMaxSm + 1];
  const int pairs = p.batch * p.n_kv;
  constexpr int A = kTileCost;
  const int B = p.item_cost;
  for (int b = threadIdx.x; b < p.batch; b += blockDim.x) {
    const Range r = seq_range(p, b);
    p.qstart[b] = r.start;
    p.lens_new[b] = r.ok ? r.end : r.start;
  }
  for (int c = threadIdx.x; c <= p.n_sm; c += blockDim.x) s_first[c] = INT_MAX;
  if (threadIdx.x == 0) s_merge = 0;
  // each thread takes a contiguous run of pairs, so prefix sums over threads follow the
  // stream order; a range of t > 0 tiles costs B + A t
  const int per = (pairs + (int)blockDim.x - 1) / (int)blockDim.x;
  const int u0 = min(pairs, (int)threadIdx.x * per), u1 = min(pairs, u0 + per);
  int mine = 0, longest = 0;
  for (int u = u0; u < u1; ++u) {
    const int t = pair_tiles(p, u);
    mine += t > 0 ? B + A * t : 0;
    longest = max(longest, t);
  }
  int W;
  const int cost0 = cta_scan(mine, tmp, &W);
  const int t_max = cta_max(longest, tmp);
  // CTAs in use: shares of at least kShareMinTiles tiles, and far enough apart that no range
  // is cut into more than max_splits items (tile centres spanning (t - 1) A cross at most
  // ceil((t - 1) A / share) share boundaries); with max_splits = 1 ranges stay whole and
  // each goes to the CTA whose share holds its middle
  const bool cut = p.max_splits >= 2;
  int share = kShareMinTiles * A + B;
  if (cut && t_max > 1) share = max(share, ((t_max - 1) * A + p.max_splits - 2) / (p.max_splits - 1));
  const int n_use = W > 0 ? max(1, min(p.n_sm, W / share)) : 0;
  // CTA c's share starts at cost y(c); owner(z) is the CTA whose share holds cost z
  auto y = [&](int c) { return (int)((long long)c * W / n_use); };
  auto owner = [&](int z) { return (int)(((long long)(z + 1) * n_use + W - 1) / W) - 1; };
  // centre of tile j of a range whose header starts at cost c0; first tile whose centre
  // is at or past cost z
  auto centre = [&](int c0, int j) { return c0 + B + A * j + A / 2; };
  auto first_tile = [&](int c0, int z) { return max(0, (z - c0 - B - A / 2 + A - 1) / A); };
  int nseg = 0;
  {
    int c0 = cost0;
    for (int u = u0; u < u1; ++u) {
      const int t = pair_tiles(p, u);
      if (t > 0) {
        nseg += cut ? owner(centre(c0, t - 1)) - owner(centre(c0, 0)) + 1 : 1;
        c0 += B + A * t;
      }
    }
  }
  int n_list;
  const int seg0 = cta_scan(nseg, tmp, &n_list);
  int c0 = cost0, i = seg0;
  for (int u = u0; u < u1; ++u) {
    const Range r = seq_range(p, u / p.n_kv);
    const int t = r.ok ? (r.end - r.lo + kTileKeys - 1) / kTileKeys : 0;
    int n = 0;
    if (t > 0) {
      const int o0 = cut ? owner(centre(c0, 0)) : owner(c0 + (B + A * t) / 2);
      const int o1 = cut ? owner(centre(c0, t - 1)) : o0;
      n = o1 - o0 + 1;
      for (int o = o0; o <= o1; ++o, ++i) {
        const int j0 = o == o0 ? 0 : first_tile(c0, y(o));
        const int j1 = o == o1 ? t : first_tile(c0, y(o + 1));
        p.items[p.n_sm + i] = make_int4(u, r.lo + j0 * kTileKeys, min(r.end, r.lo + j1 * kTileKeys),
                                        n == 1 ? -1 : o - o0);
        atomicMin(&s_first[o], i);
      }
      c0 += B + A * t;
    }
    p.splits[u] = n;
    if (n != 1)  // any order: pairs are independent
      p.merge_list[atomicAdd(&s_merge, 1)] = u | (n << kMergeCountShift);
  }
  __syncthreads();
  // items are in stream order with non-decreasing owners: CTA c starts at the first item
  // owned by c or a later CTA (a suffix minimum over the CTAs; n_sm < blockDim.x, else
  // one thread walks them)
  if ((int)blockDim.x > p.n_sm) {
    const int c = threadIdx.x;
    const int f = cta_suffix_min(c < p.n_sm ? s_first[c] : n_list, tmp);
    if (c <= p.n_sm) s_first[c] = f;
  } else if (threadIdx.x == 0) {
    s_first[p.n_sm] = n_list;
    for (int c = p.n_sm - 1; c >= 0; --c) s_first[c] = min(s_first[c], s_first[c + 1]);
  }
  if (threadIdx.x == 0) {
    *p.n_items = n_list;
    *p.n_merge = s_merge;
  }
  __syncthreads();
  for (int c = threadIdx.x; c <= p.n_sm; c += blockDim.x) {
    p.first[c] = s_first[c];
    if (c < p.n_sm)
      p.items[c] = s_first[c] < s_first[c + 1] ? p.items[p.n_sm + s_first[c + 1] - 1] : make_int4(-1, 0, 0, 0);
  }
  // the list is complete: other CTAs of the launch that builds it may read it now (they
  // only prefetch from it and never wait for this)
  __syncthreads();
  if (threadIdx.x == 0 && p.ready) {
    __threadfence();
    atomicExch(p.ready, 1);
  }
}

}  // namespace sched

// Work-list buffers and parameters of an attention call (attn_tc.cu).
sched::Params attn_sched_params(const AttnParams& a);
// Builds that work list on `s` alone (test aid); *sp receives its buffers.
cudaError_t attn_worklist_build(const AttnParams& a, cudaStream_t s, sched::Params* sp);

}  // namespace dflash
