// focus_build_index kernels: the group-sorted token index.
//
// "Focus: Learning Which Attention Pairs Matter", section 2.2: at inference
// every token goes to one group and far pairs of different groups are skipped,
// so the far part of attention only ever pairs tokens of one group.  Sorting
// tokens by (group, position) turns each group into a contiguous run of
// sorted slots, which the group pass then walks as dense tiles.
//
// Five small launches per call (two when a problem has at most 4,096 items
// and 256 groups: one block per problem does the first four steps in shared
// memory), all integer work:
//   count    per (segment, group) histogram of ids          grid (nseg, P)
//   scan     group counts, offsets, per-segment bases,
//            per-group tile bases                           grid (P)
//   scatter  stable placement: perm (slot -> position) and
//            rank (position -> slot); warp match + popc     grid (nseg, P)
//   farlen   per slot: same-group tokens at or before
//            position - w (binary search in the group run)  grid (n/256, P)
// For top-k membership the sorted items are the n_tok * k entries (token i's
// c-th group at e = i * k + c); a group never holds two entries of one token,
// so its run is still in increasing token position, and farlen compares token
// positions e >> kshift.
//   items    work list in canonical order, compacted, and
//            a longest-first schedule (stable counting sort) grid (1)
// P = B * A independent problems.
#include "common.cuh"
#include "kernels.h"

namespace focus {

namespace {

__device__ __forceinline__ int clamp_gid(int g, int K, int* err) {
  if (static_cast<unsigned>(g) >= static_cast<unsigned>(K)) {
    atomicOr(err, kErrBadGroup);
    g = g < 0 ? 0 : K - 1;
  }
  return g;
}

// Exclusive scan of one value per thread over a 1024-thread block.
__device__ int block_excl_scan(int v, int* warp_sums, int* total) {
  const int lane = lane_id(), warp = warp_id();
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_sums[lane] = s;
  }
  __syncthreads();
  int excl = x - v + (warp > 0 ? warp_sums[warp - 1] : 0);
  *total = warp_sums[31];
  __syncthreads();
  return excl;
}

// In-place exclusive scan of L <= 4 * 1024 ints in shared memory; returns the total.
__device__ int block_scan_smem(int* a, int L, int* warp_sums) {
  constexpr int kPer = 4;
  const int t = threadIdx.x;
  int v[kPer];
  int s = 0;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    int idx = t * kPer + k;
    v[k] = idx < L ? a[idx] : 0;
    s += v[k];
  }
  int total;
  int run = block_excl_scan(s, warp_sums, &total);
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    int idx = t * kPer + k;
    if (idx < L) a[idx] = run;
    run += v[k];
  }
  __syncthreads();
  return total;
}

// hist[cb] <- the number of entries in buckets above cb (an exclusive scan
// from the last bucket down), by the whole block in chunks of 4 per thread.
__device__ void bucket_starts_descending(int* hist, int nb, int* warp_sums) {
  constexpr int kPer = 4;
  int carry = 0;
  for (int base = 0; base < nb; base += kPer * blockDim.x) {
    int v[kPer];
    int s = 0;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int r = base + kPer * threadIdx.x + k;   // r-th bucket from the top
      v[k] = r < nb ? hist[nb - 1 - r] : 0;
      s += v[k];
    }
    int tot;
    int run = carry + block_excl_scan(s, warp_sums, &tot);
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int r = base + kPer * threadIdx.x + k;
      if (r < nb) hist[nb - 1 - r] = run;
      run += v[k];
    }
    carry += tot;
  }
}

__device__ __forceinline__ int upper_bound_minus1(const int* a, int len, int v) {
  // largest i in [0, len) with a[i] <= v, given a[0] <= v < a[len]
  int lo = 0, hi = len;
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (a[mid] <= v) lo = mid; else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(256) index_count_kernel(const int32_t* __restrict__ gid, int n,
                                                          int K, int nseg,
                                                          int32_t* __restrict__ segcnt, int* err) {
  extern __shared__ int hist[];
  const int p = blockIdx.y, seg = blockIdx.x;
  for (int g = threadIdx.x; g < K; g += blockDim.x) hist[g] = 0;
  __syncthreads();
  const int32_t* gp = gid + static_cast<size_t>(p) * n;
  const int start = seg * kIndexSeg, end = min(n, start + kIndexSeg);
  for (int i = start + threadIdx.x; i < end; i += blockDim.x) {
    atomicAdd(&hist[clamp_gid(__ldg(gp + i), K, err)], 1);
  }
  __syncthreads();
  int32_t* out = segcnt + (static_cast<size_t>(p) * nseg + seg) * K;
  for (int g = threadIdx.x; g < K; g += blockDim.x) out[g] = hist[g];
}

// With `staged` the [nseg][K] segment counts are first copied into shared
// memory in one coalesced pass, so the per-group walks over the segments read
// shared memory instead of issuing nseg dependent global loads each.
__global__ void __launch_bounds__(1024) index_scan_kernel(int n, int K, int nseg, int staged,
                                                          int32_t* __restrict__ segcnt,
                                                          int32_t* __restrict__ counts,
                                                          int32_t* __restrict__ offsets,
                                                          int32_t* __restrict__ tile_base) {
  extern __shared__ int sm[];
  int* cnt = sm;              // K
  int* tiles = sm + K;        // K
  int* segs = sm + 2 * K;     // [nseg][K] when staged
  __shared__ int warp_sums[32];
  const int p = blockIdx.x;
  int32_t* sc = segcnt + static_cast<size_t>(p) * nseg * K;
  if (staged) {
    for (int e = threadIdx.x; e < nseg * K; e += blockDim.x) segs[e] = sc[e];
    __syncthreads();
  }
  const int* src = staged ? segs : sc;
  for (int g = threadIdx.x; g < K; g += blockDim.x) {
    int s = 0;
    for (int seg = 0; seg < nseg; ++seg) s += src[static_cast<size_t>(seg) * K + g];
    cnt[g] = s;
    counts[static_cast<size_t>(p) * K + g] = s;
    tiles[g] = (s + kTileM - 1) / kTileM;
  }
  __syncthreads();
  int total = block_scan_smem(cnt, K, warp_sums);      // cnt -> offsets
  int ttot = block_scan_smem(tiles, K, warp_sums);     // tiles -> tile bases
  int32_t* off = offsets + static_cast<size_t>(p) * (K + 1);
  int32_t* tb = tile_base + static_cast<size_t>(p) * (K + 1);
  for (int g = threadIdx.x; g < K; g += blockDim.x) {
    off[g] = cnt[g];
    tb[g] = tiles[g];
    int run = cnt[g];
    for (int seg = 0; seg < nseg; ++seg) {
      const size_t e = static_cast<size_t>(seg) * K + g;
      const int v = src[e];
      sc[e] = run;
      run += v;
    }
  }
  if (threadIdx.x == 0) {
    off[K] = total;
    tb[K] = ttot;
  }
  (void)n;
}

__global__ void __launch_bounds__(256) index_scatter_kernel(const int32_t* __restrict__ gid, int n,
                                                            int K, int nseg,
                                                            const int32_t* __restrict__ segbase,
                                                            int32_t* __restrict__ perm,
                                                            int32_t* __restrict__ rank, int* err) {
  extern __shared__ int sm[];
  int* base = sm;                                                  // K
  uint16_t* wc = reinterpret_cast<uint16_t*>(sm + K);              // [8][K]
  const int p = blockIdx.y, seg = blockIdx.x;
  const int lane = lane_id(), warp = warp_id();
  const int32_t* gp = gid + static_cast<size_t>(p) * n;
  const int32_t* sb = segbase + (static_cast<size_t>(p) * nseg + seg) * K;
  for (int g = threadIdx.x; g < K; g += blockDim.x) base[g] = sb[g];
  for (int e = threadIdx.x; e < 8 * K; e += blockDim.x) wc[e] = 0;
  __syncthreads();
  const unsigned lt = (1u << lane) - 1u;
  const int wbeg = seg * kIndexSeg + warp * (kIndexSeg / 8);
  // per-warp group counts over this warp's 128 tokens
  for (int c = 0; c < kIndexSeg / 8; c += 32) {
    const int i = wbeg + c + lane;
    const bool valid = i < n;
    const int g = valid ? clamp_gid(__ldg(gp + i), K, err) : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, g);
    if (valid && lane == __ffs(peers) - 1) wc[warp * K + g] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  for (int g = threadIdx.x; g < K; g += blockDim.x) {
    int run = 0;
    for (int w = 0; w < 8; ++w) {
      int v = wc[w * K + g];
      wc[w * K + g] = static_cast<uint16_t>(run);
      run += v;
    }
  }
  __syncthreads();
  int32_t* pp = perm + static_cast<size_t>(p) * n;
  int32_t* rp = rank + static_cast<size_t>(p) * n;
  for (int c = 0; c < kIndexSeg / 8; c += 32) {
    const int i = wbeg + c + lane;
    const bool valid = i < n;
    const int g = valid ? clamp_gid(__ldg(gp + i), K, err) : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, g);
    if (valid) {
      const int slot = base[g] + wc[warp * K + g] + __popc(peers & lt);
      pp[slot] = i;
      rp[i] = slot;
    }
    __syncwarp();
    if (valid && lane == __ffs(peers) - 1) wc[warp * K + g] += __popc(peers);
    __syncwarp();
  }
}

__global__ void __launch_bounds__(256) index_farlen_kernel(int n, int K, int w_eff, int kshift,
                                                           const int32_t* __restrict__ offsets,
                                                           const int32_t* __restrict__ perm,
                                                           int32_t* __restrict__ farlen_tok,
                                                           int32_t* __restrict__ farlen_slot) {
  extern __shared__ int offs[];  // K + 1
  const int p = blockIdx.y;
  const int32_t* op = offsets + static_cast<size_t>(p) * (K + 1);
  for (int g = threadIdx.x; g <= K; g += blockDim.x) offs[g] = op[g];
  __syncthreads();
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= n) return;
  const int32_t* pp = perm + static_cast<size_t>(p) * n;
  const int item = pp[s];
  const int pos = item >> kshift;
  const int g = upper_bound_minus1(offs, K, s);
  // members of g at slots [offs[g], s) have positions < pos; count those
  // with position <= pos - w_eff, i.e. < target
  const int target = pos - w_eff + 1;
  // positions rise along the group's slots, so at most w_eff - 1 members
  // before slot s lie at or after target: the answer is within w_eff - 1
  // slots of s
  int lo = max(offs[g], s - w_eff + 1), hi = s;   // first slot in [lo, hi) whose position >= target
  while (lo < hi) {
    int mid = (lo + hi) >> 1;
    if ((__ldg(pp + mid) >> kshift) < target) lo = mid + 1; else hi = mid;
  }
  const int fl = lo - offs[g];
  farlen_slot[static_cast<size_t>(p) * n + s] = fl;
  farlen_tok[static_cast<size_t>(p) * n + item] = fl;
}

__global__ void __launch_bounds__(1024) index_items_kernel(
    int P, int A, int n, int K, int staged, int cstaged, const int32_t* __restrict__ counts,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ tile_base,
    const int32_t* __restrict__ farlen_slot, focus_item_t* __restrict__ items,
    int32_t* __restrict__ cost, int32_t* __restrict__ order, int32_t* __restrict__ n_items,
    int max_items, int* err) {
  extern __shared__ int sm[];
  int* pbase = sm;                 // P + 1
  int* hist = sm + P + 1;          // nb + 1
  __shared__ int warp_sums[32];
  const int nb = (n + kTileN - 1) / kTileN + 1;   // cost buckets 0..nb-1
  // with `staged` every problem's tile bases are copied to shared memory, so
  // each candidate's search over them reads no global memory
  int* tbs = hist + nb + 1;        // [P][K + 1] when staged
  // with `cstaged` the items' cost buckets are also kept in shared memory, so
  // the ordering loop below reads no global memory
  int* cs = tbs + (staged ? P * (K + 1) : 0);   // [max_items] when cstaged
  if (staged) {
    for (int e = threadIdx.x; e < P * (K + 1); e += blockDim.x) tbs[e] = tile_base[e];
  }
  if (threadIdx.x == 0) {
    int run = 0;
    for (int p = 0; p < P; ++p) {
      pbase[p] = run;
      run += tile_base[static_cast<size_t>(p) * (K + 1) + K];
    }
    pbase[P] = run;
  }
  for (int c = threadIdx.x; c < nb; c += blockDim.x) hist[c] = 0;
  __syncthreads();
  const int total = pbase[P];
  int out = 0;
  for (int c0 = 0; c0 < total; c0 += blockDim.x) {
    const int c = c0 + threadIdx.x;
    int flag = 0;
    focus_item_t it{};
    if (c < total) {
      const int p = upper_bound_minus1(pbase, P, c);
      const int t = c - pbase[p];
      const int32_t* tb = (staged ? tbs : tile_base) + static_cast<size_t>(p) * (K + 1);
      // group of candidate tile t: largest g with tb[g] <= t (tb[K] > t)
      int lo = 0, hi = K;
      while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (tb[mid] <= t) lo = mid; else hi = mid;
      }
      const int g = lo;
      const int tt = t - tb[g];
      const int off = offsets[static_cast<size_t>(p) * (K + 1) + g];
      const int cnt = counts[static_cast<size_t>(p) * K + g];
      it.b = p / A;
      it.a = p % A;
      it.g = g;
      it.row0 = off + tt * kTileM;
      it.rows = min(kTileM, cnt - tt * kTileM);
      it.key0 = off;
      if (it.rows <= 0) {
        atomicOr(err, kErrInternal);
      } else {
        it.keys = farlen_slot[static_cast<size_t>(p) * n + it.row0 + it.rows - 1];
        flag = it.keys > 0;
      }
    }
    int tot;
    const int pos = block_excl_scan(flag, warp_sums, &tot);
    if (flag && out + pos < max_items) {
      items[out + pos] = it;
      const int cb = (it.keys + kTileN - 1) / kTileN;
      cost[out + pos] = cb;
      if (cstaged) cs[out + pos] = cb;
      atomicAdd(&hist[cb], 1);
    }
    out += tot;
  }
  if (out > max_items) {
    if (threadIdx.x == 0) atomicOr(err, kErrInternal);
    out = max_items;
  }
  __syncthreads();
  bucket_starts_descending(hist, nb, warp_sums);   // start of each cost bucket, costliest first
  if (threadIdx.x == 0) *n_items = out;
  __syncthreads();
  if (warp_id() == 0) {
    const int lane = lane_id();
    const unsigned lt = (1u << lane) - 1u;
    const int* csrc = cstaged ? cs : cost;
    for (int c0 = 0; c0 < out; c0 += 32) {
      const int c = c0 + lane;
      const int cb = c < out ? csrc[c] : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, cb);
      if (c < out) order[hist[cb] + __popc(peers & lt)] = c;
      __syncwarp();
      if (c < out && lane == __ffs(peers) - 1) hist[cb] += __popc(peers);
      __syncwarp();
    }
  }
}

// Small problems (n <= kSmallN items, K <= kSmallK groups; one block per
// problem costs about 2 ns per item, so above a few thousand items the
// general kernels are faster): count, scan,
// stable scatter and far lengths of one problem in one block, all in shared
// memory, so the index is two launches (this and the work list) instead of
// five.  The results are the same arrays the general kernels write: tokens
// placed in order of position within each group (chunks of 1,024 in order,
// warps in order within a chunk, lanes in order within a warp).
constexpr int kSmallN = 4096;
constexpr int kSmallK = 256;

__global__ void __launch_bounds__(1024, 1) index_small_kernel(const int32_t* __restrict__ gid, int n, int K,
                                                           int w_eff, int kshift,
                                                           int32_t* __restrict__ counts,
                                                           int32_t* __restrict__ offsets,
                                                           int32_t* __restrict__ tile_base,
                                                           int32_t* __restrict__ perm,
                                                           int32_t* __restrict__ rank,
                                                           int32_t* __restrict__ farlen_tok,
                                                           int32_t* __restrict__ farlen_slot, int* err) {
  extern __shared__ int sm[];
  int* gs = sm;                 // [n] group of each item
  int* ps = gs + n;             // [n] perm
  int* cnt = ps + n;            // [K] counts, then offsets
  int* tiles = cnt + K;         // [K] tile counts, then tile bases
  int* run = tiles + K;         // [K] next slot of each group
  int* wc = run + K;            // [32][K + 1] per-warp counts of a chunk, then their prefixes
  const int Kp = K + 1;         // row stride: a group's 32 warp entries fall in 32 banks
  __shared__ int warp_sums[32];
  const int p = blockIdx.x;
  const int lane = lane_id(), warp = warp_id();
  const unsigned lt = (1u << lane) - 1u;
  const int32_t* gp = gid + static_cast<size_t>(p) * n;
  for (int g = threadIdx.x; g < K; g += blockDim.x) cnt[g] = 0;
  for (int e = threadIdx.x; e < 32 * Kp; e += blockDim.x) wc[e] = 0;
  __syncthreads();
  // all of this thread's ids are requested before the first is used
#pragma unroll 8
  for (int i = threadIdx.x; i < n; i += blockDim.x) gs[i] = __ldg(gp + i);
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int g = clamp_gid(gs[i], K, err);
    gs[i] = g;
    atomicAdd(&cnt[g], 1);
  }
  __syncthreads();
  for (int g = threadIdx.x; g < K; g += blockDim.x) {
    counts[static_cast<size_t>(p) * K + g] = cnt[g];
    tiles[g] = (cnt[g] + kTileM - 1) / kTileM;
  }
  __syncthreads();
  const int total = block_scan_smem(cnt, K, warp_sums);    // cnt -> offsets
  const int ttot = block_scan_smem(tiles, K, warp_sums);   // tiles -> tile bases
  int32_t* off = offsets + static_cast<size_t>(p) * (K + 1);
  int32_t* tb = tile_base + static_cast<size_t>(p) * (K + 1);
  for (int g = threadIdx.x; g < K; g += blockDim.x) {
    off[g] = cnt[g];
    tb[g] = tiles[g];
    run[g] = cnt[g];
  }
  if (threadIdx.x == 0) {
    off[K] = total;
    tb[K] = ttot;
  }
  __syncthreads();
  // stable placement, 1,024 items per chunk
  int32_t* pp = perm + static_cast<size_t>(p) * n;
  int32_t* rp = rank + static_cast<size_t>(p) * n;
  for (int c0 = 0; c0 < n; c0 += blockDim.x) {
    const int i = c0 + threadIdx.x;
    const bool valid = i < n;
    const int g = valid ? gs[i] : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, g);
    if (valid && lane == __ffs(peers) - 1) wc[warp * Kp + g] = __popc(peers);
    __syncthreads();
    // per group, a warp scans the 32 warp counts (lane = warp of the chunk)
    for (int gg = warp; gg < K; gg += 32) {
      const int v = wc[lane * Kp + gg];
      int x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      const int base = run[gg];
      wc[lane * Kp + gg] = base + x - v;
      __syncwarp();
      if (lane == 31) run[gg] = base + x;
    }
    __syncthreads();
    if (valid) {
      const int slot = wc[warp * Kp + g] + __popc(peers & lt);
      ps[slot] = i;
      pp[slot] = i;
      rp[i] = slot;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < 32 * Kp; e += blockDim.x) wc[e] = 0;
    __syncthreads();
  }
  // far lengths: same-group items at positions <= pos - w_eff, searched
  // within w_eff - 1 slots before s (positions rise along a group's slots)
  for (int sl = threadIdx.x; sl < n; sl += blockDim.x) {
    const int item = ps[sl];
    const int pos = item >> kshift;
    const int g = gs[item];
    const int target = pos - w_eff + 1;
    int lo = max(cnt[g], sl - w_eff + 1), hi = sl;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if ((ps[mid] >> kshift) < target) lo = mid + 1; else hi = mid;
    }
    const int fl = lo - cnt[g];
    farlen_slot[static_cast<size_t>(p) * n + sl] = fl;
    farlen_tok[static_cast<size_t>(p) * n + item] = fl;
  }
}

size_t small_smem(int n, int K) {
  return (2 * static_cast<size_t>(n) + 3 * static_cast<size_t>(K) + 32 * (static_cast<size_t>(K) + 1)) * sizeof(int);
}

// Split top-2 index, far prefixes: for sorted slot s of entry e (token
// i = e >> 1) in virtual group v = g * K + o, and each other group o' != g
// (column j = o' - (o' > g)), the members of sub-run (g, o') at positions
// <= i - w, or 0 when o' == o and o < g (that pair's pass is group o's).
// m = 2n slots per problem; Kv = K * K virtual groups.
__global__ void __launch_bounds__(256) index_farlen_split_kernel(int m, int K, int w_eff,
                                                                 const int32_t* __restrict__ offsets,
                                                                 const int32_t* __restrict__ perm,
                                                                 int32_t* __restrict__ farlen_sub,
                                                                 int32_t* __restrict__ farlen_tok,
                                                                 int32_t* __restrict__ farlen_slot) {
  extern __shared__ int offs[];  // K * K + 1
  const int p = blockIdx.y;
  const int Kv = K * K;
  const int32_t* op = offsets + static_cast<size_t>(p) * (Kv + 1);
  for (int v = threadIdx.x; v <= Kv; v += blockDim.x) offs[v] = op[v];
  __syncthreads();
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= m) return;
  const int32_t* pp = perm + static_cast<size_t>(p) * m;
  const int e = pp[s];
  const int pos = e >> 1;
  const int v = upper_bound_minus1(offs, Kv, s);
  const int g = v / K, o = v - g * K;
  const int target = pos - w_eff + 1;   // count members with position < target
  int32_t* fs = farlen_sub + (static_cast<size_t>(p) * m + s) * (K - 1);
  int total = 0;
  for (int o2 = 0; o2 < K; ++o2) {
    if (o2 == g) continue;
    const int j = o2 < g ? o2 : o2 - 1;
    int fl = 0;
    if (!(o2 == o && o < g)) {
      const int v2 = g * K + o2;
      int lo = offs[v2], hi = offs[v2 + 1];    // first slot whose position >= target
      const int base = lo;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if ((__ldg(pp + mid) >> 1) < target) lo = mid + 1; else hi = mid;
      }
      fl = lo - base;
    }
    fs[j] = fl;
    total += fl;
  }
  farlen_slot[static_cast<size_t>(p) * m + s] = total;
  farlen_tok[static_cast<size_t>(p) * m + e] = total;
}

// Split work list: candidates (problem, row tile of a virtual group) in
// canonical order; an item when the tile's last row has far keys in any of
// its group's sub-runs (keys = their total, key0 = the group's first slot;
// the attention kernel walks the sub-runs from offsets and farlen_sub); then
// the same compaction and longest-first schedule as index_items_kernel.
// item.g = virtual group.
__global__ void __launch_bounds__(1024) index_items_split_kernel(
    int P, int A, int m, int K, int cstaged, const int32_t* __restrict__ counts,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ tile_base,
    const int32_t* __restrict__ farlen_sub, focus_item_t* __restrict__ items,
    int32_t* __restrict__ cost, int32_t* __restrict__ order, int32_t* __restrict__ n_items,
    int max_items, int* err) {
  extern __shared__ int sm[];
  int* pbase = sm;                 // P + 1
  int* hist = sm + P + 1;          // nb + 1
  __shared__ int warp_sums[32];
  const int Kv = K * K, nsub = K - 1;
  // cost buckets 0..nb-1: a tile's keys over its sub-runs stay below m + K * kTileN
  const int nb = (m + kTileN - 1) / kTileN + K + 1;
  int* cs = hist + nb + 1;         // [max_items] cost buckets when cstaged
  if (threadIdx.x == 0) {
    int run = 0;
    for (int p = 0; p < P; ++p) {
      pbase[p] = run;
      run += tile_base[static_cast<size_t>(p) * (Kv + 1) + Kv];
    }
    pbase[P] = run;
  }
  for (int c = threadIdx.x; c < nb; c += blockDim.x) hist[c] = 0;
  __syncthreads();
  const int total = pbase[P];
  int out = 0;
  for (int c0 = 0; c0 < total; c0 += blockDim.x) {
    const int c = c0 + threadIdx.x;
    int flag = 0;
    focus_item_t it{};
    if (c < total) {
      const int p = upper_bound_minus1(pbase, P, c);
      const int t = c - pbase[p];
      const int32_t* tb = tile_base + static_cast<size_t>(p) * (Kv + 1);
      int lo = 0, hi = Kv;        // virtual group of tile t: largest v with tb[v] <= t
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(tb + mid) <= t) lo = mid; else hi = mid;
      }
      const int v = lo, g = v / K;
      const int tt = t - tb[v];
      const int32_t* op = offsets + static_cast<size_t>(p) * (Kv + 1);
      const int off = op[v];
      const int cnt = counts[static_cast<size_t>(p) * Kv + v];
      it.b = p / A;
      it.a = p % A;
      it.g = v;
      it.row0 = off + tt * kTileM;
      it.rows = min(kTileM, cnt - tt * kTileM);
      it.key0 = op[g * K];
      it.pad = 0;
      if (it.rows <= 0) {
        atomicOr(err, kErrInternal);
      } else {
        const int32_t* fl = farlen_sub + (static_cast<size_t>(p) * m + it.row0 + it.rows - 1) * nsub;
        int keys = 0;
        for (int j = 0; j < nsub; ++j) keys += fl[j];
        it.keys = keys;
        flag = keys > 0;
      }
    }
    int tot;
    const int pos = block_excl_scan(flag, warp_sums, &tot);
    if (flag && out + pos < max_items) {
      items[out + pos] = it;
      const int cb = (it.keys + kTileN - 1) / kTileN;
      cost[out + pos] = cb;
      if (cstaged) cs[out + pos] = cb;
      atomicAdd(&hist[cb], 1);
    }
    out += tot;
  }
  if (out > max_items) {
    if (threadIdx.x == 0) atomicOr(err, kErrInternal);
    out = max_items;
  }
  __syncthreads();
  bucket_starts_descending(hist, nb, warp_sums);   // start of each cost bucket, costliest first
  if (threadIdx.x == 0) *n_items = out;
  __syncthreads();
  if (warp_id() == 0) {
    const int lane = lane_id();
    const unsigned lt = (1u << lane) - 1u;
    const int* csrc = cstaged ? cs : cost;
    for (int c0 = 0; c0 < out; c0 += 32) {
      const int c = c0 + lane;
      const int cb = c < out ? csrc[c] : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, cb);
      if (c < out) order[hist[cb] + __popc(peers & lt)] = c;
      __syncwarp();
      if (c < out && lane == __ffs(peers) - 1) hist[cb] += __popc(peers);
      __syncwarp();
    }
  }
}

// Shared-memory staging limits: the scan's [nseg][K] segment counts and the
// work-list kernel's [P][K + 1] tile bases.
constexpr int kScanStageInts = 16384;    // 64 KB
constexpr int kItemsStageInts = 8192;    // 32 KB
constexpr int kCostStageInts = 8192;     // 32 KB: the work list's cost buckets

int scan_staged(int nseg, int K) {
  return static_cast<long long>(nseg) * K <= kScanStageInts ? 1 : 0;
}
size_t scan_smem(int nseg, int K, int staged) {
  return (2 * static_cast<size_t>(K) + (staged ? static_cast<size_t>(nseg) * K : 0)) * sizeof(int);
}

}  // namespace

cudaError_t launch_build_index_split(const IndexLaunch& L, int K, int32_t* farlen_sub, cudaStream_t st) {
  const int P = L.P;
  const int Kv = L.K;            // K * K virtual groups
  if (K < 2 || Kv != K * K || L.kshift != 1) return cudaErrorInvalidValue;
  const int nseg = (L.n + kIndexSeg - 1) / kIndexSeg;
  index_count_kernel<<<dim3(nseg, P), 256, static_cast<size_t>(Kv) * sizeof(int), st>>>(
      L.gid, L.n, Kv, nseg, L.segcnt, L.err);
  const int staged_s = scan_staged(nseg, Kv);
  index_scan_kernel<<<P, 1024, scan_smem(nseg, Kv, staged_s), st>>>(
      L.n, Kv, nseg, staged_s, L.segcnt, L.counts, L.offsets, L.tile_base);
  index_scatter_kernel<<<dim3(nseg, P), 256, static_cast<size_t>(Kv) * sizeof(int) + 8 * static_cast<size_t>(Kv) * 2,
                         st>>>(L.gid, L.n, Kv, nseg, L.segcnt, L.perm, L.rank, L.err);
  index_farlen_split_kernel<<<dim3((L.n + 255) / 256, P), 256, static_cast<size_t>(Kv + 1) * sizeof(int), st>>>(
      L.n, K, L.w_eff, L.offsets, L.perm, farlen_sub, L.farlen_tok, L.farlen_slot);
  const int nb = (L.n + kTileN - 1) / kTileN + K + 1;
  const int cst = L.max_items <= kCostStageInts ? 1 : 0;
  index_items_split_kernel<<<1, 1024, static_cast<size_t>(P + 1 + nb + (cst ? L.max_items : 0)) * sizeof(int), st>>>(
      P, L.A, L.n, K, cst, L.counts, L.offsets, L.tile_base, farlen_sub, L.items, L.cost, L.order, L.n_items,
      L.max_items, L.err);
  return cudaGetLastError();
}

cudaError_t launch_build_index(const IndexLaunch& L, cudaStream_t st) {
  const int P = L.P;
  const int nseg = (L.n + kIndexSeg - 1) / kIndexSeg;
  const bool small = L.n <= kSmallN && L.K <= kSmallK;
  if (small) {
    index_small_kernel<<<P, 1024, small_smem(L.n, L.K), st>>>(L.gid, L.n, L.K, L.w_eff, L.kshift, L.counts,
                                                               L.offsets, L.tile_base, L.perm, L.rank,
                                                               L.farlen_tok, L.farlen_slot, L.err);
  } else {
    const size_t sm_count = static_cast<size_t>(L.K) * sizeof(int);
    index_count_kernel<<<dim3(nseg, P), 256, sm_count, st>>>(L.gid, L.n, L.K, nseg, L.segcnt, L.err);
    const int staged_s = scan_staged(nseg, L.K);
    index_scan_kernel<<<P, 1024, scan_smem(nseg, L.K, staged_s), st>>>(
        L.n, L.K, nseg, staged_s, L.segcnt, L.counts, L.offsets, L.tile_base);
    const size_t sm_scatter = static_cast<size_t>(L.K) * sizeof(int) + 8 * static_cast<size_t>(L.K) * 2;
    index_scatter_kernel<<<dim3(nseg, P), 256, sm_scatter, st>>>(L.gid, L.n, L.K, nseg, L.segcnt,
                                                                  L.perm, L.rank, L.err);
    const size_t sm_far = static_cast<size_t>(L.K + 1) * sizeof(int);
    index_farlen_kernel<<<dim3((L.n + 255) / 256, P), 256, sm_far, st>>>(
        L.n, L.K, L.w_eff, L.kshift, L.offsets, L.perm, L.farlen_tok, L.farlen_slot);
  }
  const int nb = (L.n + kTileN - 1) / kTileN + 1;
  const long long tb_ints = static_cast<long long>(P) * (L.K + 1);
  const int staged_i = tb_ints <= kItemsStageInts ? 1 : 0;
  const int cst = L.max_items <= kCostStageInts ? 1 : 0;
  const size_t sm_items =
      static_cast<size_t>(P + 1 + nb + (staged_i ? tb_ints : 0) + (cst ? L.max_items : 0)) * sizeof(int);
  index_items_kernel<<<1, 1024, sm_items, st>>>(P, L.A, L.n, L.K, staged_i, cst, L.counts, L.offsets,
                                                L.tile_base, L.farlen_slot, L.items, L.cost,
                                                L.order, L.n_items, L.max_items, L.err);
  return cudaGetLastError();
}

cudaError_t setup_index_kernels() {
  // dynamic shared memory above 48 KB for the largest K and n
  cudaError_t e = cudaFuncSetAttribute(index_scatter_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kMaxK * 4 + 8 * kMaxK * 2);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(index_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(small_smem(kSmallN, kSmallK)));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(index_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (2 * kMaxK + kScanStageInts) * 4);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(index_items_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           160 * 1024 + (kItemsStageInts + kCostStageInts) * 4);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(index_items_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           160 * 1024 + kCostStageInts * 4);
  return e;
}

}  // namespace focus
