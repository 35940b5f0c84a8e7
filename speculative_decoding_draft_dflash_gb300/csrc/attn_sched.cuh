// Work list of the tensor-core block attention, computed by one CTA.
//
// For every sequence b the block occupies positions start .. start + bs - 1,
// start = lens[b] plus the rows a KV inject issued in the same call appended
// (DFlash KV Injection Walkthrough, Step 7: the cache grows by the new context
// rows, then the block follows them). The keys a query of the block sees are
// [lo, start + bs): the whole prefix, or the last W positions under a sliding
// window of W (the window reading of the hybrid layers). Each (sequence, KV
// head) pair's key range is cut into items of about equal tile counts; the
// items are listed largest first, which the attention CTAs then take in order
// from an atomic counter.
//
// The same pass records, per sequence, the block start (read by the attention
// for the window test) and the cache length after the call, which the combine
// kernel writes back once the attention has finished with the old lengths.
#pragma once

#include "dflash_internal.cuh"

namespace dflash {
namespace sched {

constexpr int kTileKeys = 128;     // keys per attention tile
constexpr int kItemMinTiles = 4;   // smallest item worth a pipeline ramp
constexpr int kMaxClass = 64;      // item sizes in tiles are bucketed up to this

struct Params {
  const int32_t* lens;      // [batch] lengths before the call
  const int32_t* pre_rows;  // cu_rows [batch + 1] of rows injected in the same call, or null
  int pre_M;                // row count of that inject
  int4* items;              // {pair, k_begin, k_end, split (-1 = whole range)}
  int* n_items;
  int* next_item;
  int* splits;              // [pair]: items of the pair (0 = refused sequence)
  int* merge_list;          // pairs whose rows the combine writes (split or refused),
  int* n_merge;             //   and their count
  int* ready;               // set to 1 once the list is complete (the attention clears it)
  int32_t* qstart;          // [batch]: first position of the block
  int32_t* lens_new;        // [batch]: length after the call
  int batch, n_kv, bs, window, capacity, table_len, max_splits, n_sm;
  int align;                // key ranges start on multiples of this (paged cache: a page)
};

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

__device__ __forceinline__ int cta_sum(int v, int* tmp) {
  v = __reduce_add_sync(0xffffffffu, v);
  if ((threadIdx.x & 31) == 0) tmp[threadIdx.x >> 5] = v;
  __syncthreads();
  int t = 0;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += tmp[i];
  __syncthreads();
  return t;
}

// Three sums at once (tmp: 3 x 32 ints); every thread gets the totals in v.
__device__ __forceinline__ void cta_sum3(int (&v)[3], int* tmp) {
  const int w = threadIdx.x >> 5, nw = (int)(blockDim.x >> 5);
  for (int i = 0; i < 3; ++i) {
    const int x = __reduce_add_sync(0xffffffffu, v[i]);
    if ((threadIdx.x & 31) == 0) tmp[i * 32 + w] = x;
  }
  __syncthreads();
  for (int i = 0; i < 3; ++i) {
    int t = 0;
    for (int j = 0; j < nw; ++j) t += tmp[i * 32 + j];
    v[i] = t;
  }
  __syncthreads();
}

// Run by every thread of one CTA (blockDim.x a multiple of 32, at least kMaxClass + 1).
inline __device__ void build(const Params& p) {
  __shared__ int tmp[96];
  __shared__ int s_class_base[kMaxClass + 1];
  __shared__ int s_class_cnt[kMaxClass + 1];
  __shared__ int s_merge;
  const int pairs = p.batch * p.n_kv;
  // total tiles, then the item size (below); at least kItemMinTiles tiles per item and
  // never more than max_splits items per range
  int mine = 0;
  for (int b = threadIdx.x; b < p.batch; b += blockDim.x) {
    const Range r = seq_range(p, b);
    if (r.ok) mine += p.n_kv * ((r.end - r.lo + kTileKeys - 1) / kTileKeys);
    p.qstart[b] = r.start;
    p.lens_new[b] = r.ok ? r.end : r.start;
  }
  const int total_tiles = cta_sum(mine, tmp);
  // Item size: about F items per SM for F = 2, 3 or 4. Items are taken greedily, largest
  // first, so the finish is even when the item count fills whole waves of n_sm CTAs; with
  // equal sequences (one long context, equal windows) a count just past a wave leaves most
  // SMs idle at the end. Take the smallest F whose count fills its last wave within 5% of
  // the best of the three.
  int cand[3], cnt[3] = {0, 0, 0};
  for (int f = 0; f < 3; ++f)
    cand[f] = max(kItemMinTiles, (total_tiles + (f + 2) * p.n_sm - 1) / ((f + 2) * p.n_sm));
  for (int b = threadIdx.x; b < p.batch; b += blockDim.x) {
    const Range r = seq_range(p, b);
    if (!r.ok) continue;
    const int t = (r.end - r.lo + kTileKeys - 1) / kTileKeys;
    for (int f = 0; f < 3; ++f) cnt[f] += p.n_kv * min(p.max_splits, (t + cand[f] - 1) / cand[f]);
  }
  cta_sum3(cnt, tmp);
  float fill[3], best = 0.f;
  for (int f = 0; f < 3; ++f) {
    const int waves = (cnt[f] + p.n_sm - 1) / p.n_sm;
    fill[f] = waves > 0 ? (float)cnt[f] / (float)(waves * p.n_sm) : 1.f;
    best = fmaxf(best, fill[f]);
  }
  int item_tiles = cand[2];
  for (int f = 2; f >= 0; --f)
    if (fill[f] >= best - 0.05f) item_tiles = cand[f];
  if (threadIdx.x <= kMaxClass) s_class_cnt[threadIdx.x] = 0;
  if (threadIdx.x == 0) {
    *p.next_item = 0;
    s_merge = 0;
  }
  __syncthreads();
  // A range of t tiles becomes n = ceil(t / item_tiles) items of floor / ceil(t / n) tiles;
  // count the items of each size
  for (int pr = threadIdx.x; pr < pairs; pr += blockDim.x) {
    const Range r = seq_range(p, pr / p.n_kv);
    int n = 0;
    if (r.ok) {
      const int t = (r.end - r.lo + kTileKeys - 1) / kTileKeys;
      n = (t + item_tiles - 1) / item_tiles;
      if (n > p.max_splits) n = p.max_splits;
      const int small = t / n, big_cnt = t - small * n;  // big_cnt items of small + 1 tiles
      if (big_cnt) atomicAdd(&s_class_cnt[min(small + 1, kMaxClass)], big_cnt);
      if (n - big_cnt) atomicAdd(&s_class_cnt[min(small, kMaxClass)], n - big_cnt);
    }
    p.splits[pr] = n;
    if (n != 1) p.merge_list[atomicAdd(&s_merge, 1)] = pr;  // any order: pairs are independent
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int c = kMaxClass; c >= 0; --c) {  // largest items first
      s_class_base[c] = acc;
      acc += s_class_cnt[c];
    }
    *p.n_items = acc;
    *p.n_merge = s_merge;
  }
  __syncthreads();
  if (threadIdx.x <= kMaxClass) s_class_cnt[threadIdx.x] = 0;
  __syncthreads();
  for (int pr = threadIdx.x; pr < pairs; pr += blockDim.x) {
    const int n = p.splits[pr];
    if (n == 0) continue;
    const Range r = seq_range(p, pr / p.n_kv);
    const int t = (r.end - r.lo + kTileKeys - 1) / kTileKeys;
    const int small = t / n, big_cnt = t - small * n;
    int k = r.lo;
    for (int s = 0; s < n; ++s) {
      const int tiles = small + (s < big_cnt ? 1 : 0);
      const int c = min(tiles, kMaxClass);
      const int slot = s_class_base[c] + atomicAdd(&s_class_cnt[c], 1);
      const int k1 = min(r.end, k + tiles * kTileKeys);
      p.items[slot] = make_int4(pr, k, k1, n == 1 ? -1 : s);
      k = k1;
    }
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

}  // namespace dflash
