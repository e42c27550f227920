// Top-2 group membership: the kernels that turn two memberships per token into
// one far partial per token.
//
// "Focus: Learning Which Attention Pairs Matter", section 2.2: at inference
// each token goes to its top-k groups; "Why Attend to Everything? Focus is the
// Key", section 2.3 runs the method with K = 4, k = 2.  A far pair (j <= i - w)
// is kept when the two tokens' group sets meet, and softmax stays exact over
// the kept pairs, each counted once.
//
// The group pass runs over entries (token i's c-th group, e = 2i + c), so it
// produces, per token, one partial over the far keys of each of its groups.  A
// key that shares both groups with the query appears in both: those keys are
// exactly the earlier far members of the query's group pair {a, b}, which a
// second group pass over pair ids computes as a partial of its own.  With
// weights w = exp(lse - M), the far softmax over the union is
//   O = (w_a O_a + w_b O_b - w_ab O_ab) / (w_a + w_b - w_ab),
//   lse = M + log(w_a + w_b - w_ab).
// The pair keys are a subset of each group's keys, so w_ab <= min(w_a, w_b)
// and the denominator is at least max(w_a, w_b): it never cancels, and the
// result's error is at most three roundings of the stored partials.
//
// For small K the index can be split instead (memberships sorted by group,
// then the token's other group, then position): the entry of the larger of
// two shared groups skips the sub-run of the other one, so every far pair is
// visited once, there is no pair partial, and the merge is the plain
// log-sum-exp of the two entry partials.
#include "common.cuh"
#include "kernels.h"

namespace focus {
namespace {

__global__ void __launch_bounds__(256) pair_ids_kernel(const int2* __restrict__ gid2, long long total,
                                                       int K, int32_t* __restrict__ pair_gid,
                                                       int* err) {
  for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t < total;
       t += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int2 g = __ldg(gid2 + t);
    int lo = min(g.x, g.y), hi = max(g.x, g.y);
    if (lo < 0 || hi >= K || lo == hi) {
      // not two distinct groups in [0, K): flag it and file the token under
      // pair 0 so every later index stays in bounds
      atomicOr(err, kErrBadGroup);
      lo = 0;
      hi = 1;
    }
    // pairs {lo, hi} numbered row by row: (0,1), (0,2), ..., (0,K-1), (1,2), ...
    pair_gid[t] = lo * K - lo * (lo + 1) / 2 + (hi - lo - 1);
  }
}

// Virtual group ids of the split index: entry 2i + c of token i with groups
// (g_0, g_1) gets g_c * K + g_(1-c).
__global__ void __launch_bounds__(256) split_ids_kernel(const int2* __restrict__ gid2, long long total,
                                                        int K, int2* __restrict__ vg, int* err) {
  for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t < total;
       t += static_cast<long long>(gridDim.x) * blockDim.x) {
    int2 g = __ldg(gid2 + t);
    if (g.x < 0 || g.x >= K || g.y < 0 || g.y >= K || g.x == g.y) {
      // not two distinct groups in [0, K): flag it and file the token under
      // groups 0 and 1 so every later index stays in bounds
      atomicOr(err, kErrBadGroup);
      g = make_int2(0, 1);
    }
    vg[t] = make_int2(g.x * K + g.y, g.y * K + g.x);
  }
}

__global__ void __launch_bounds__(256) far_any_kernel(const int2* __restrict__ farlen_entry,
                                                      long long total, int32_t* __restrict__ far_any) {
  for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t < total;
       t += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int2 f = __ldg(farlen_entry + t);
    far_any[t] = (f.x > 0 || f.y > 0) ? 1 : 0;
  }
}

template <typename T>
struct Vec8;   // eight elements of one row, as one 16- or two 16-byte words
template <>
struct Vec8<__nv_bfloat16> {
  uint4 u;
  __device__ __forceinline__ void load(const void* base, size_t off) {
    u = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + off));
  }
  __device__ __forceinline__ float get(int e) const {
    const uint32_t w = (&u.x)[e >> 1];
    return __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
  }
  __device__ __forceinline__ void set_all(const float* f) {
    u.x = pack_bf16x2(f[0], f[1]);
    u.y = pack_bf16x2(f[2], f[3]);
    u.z = pack_bf16x2(f[4], f[5]);
    u.w = pack_bf16x2(f[6], f[7]);
  }
  __device__ __forceinline__ void store(void* base, size_t off) const {
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + off) = u;
  }
};
template <>
struct Vec8<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const void* base, size_t off) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + off);
    a = __ldg(p);
    b = __ldg(p + 1);
  }
  __device__ __forceinline__ float get(int e) const {
    const float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    return f[e];
  }
  __device__ __forceinline__ void set_all(const float* f) {
    a = make_float4(f[0], f[1], f[2], f[3]);
    b = make_float4(f[4], f[5], f[6], f[7]);
  }
  __device__ __forceinline__ void store(void* base, size_t off) const {
    float4* p = reinterpret_cast<float4*>(static_cast<float*>(base) + off);
    p[0] = a;
    p[1] = b;
  }
};

// One thread per eight elements of a query row (zq, i); d / 8 threads per row.
template <typename T>
__global__ void __launch_bounds__(256) topk_merge_kernel(MergeLaunch L, long long rows) {
  const int per_row = L.d / 8;
  const long long total = rows * per_row;
  const size_t m = 2 * static_cast<size_t>(L.n);
  for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t < total;
       t += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = t / per_row;
    const int part = static_cast<int>(t % per_row);
    const int i = static_cast<int>(row % L.n);
    const int zq = static_cast<int>(row / L.n);
    const int b = zq / L.H, h = zq % L.H;
    const int kv = (h * L.H_kv) / L.H;
    const size_t p = static_cast<size_t>(b) * L.A + (L.A == 1 ? 0 : kv);
    const bool fa = __ldg(L.farlen_entry + p * m + 2 * i) > 0;
    const bool fb = __ldg(L.farlen_entry + p * m + 2 * i + 1) > 0;
    if (!fa && !fb) continue;            // no far keys: the local pass reads nothing here
    // a consistent index has pair far keys only where both groups have some;
    // the split index visits every far pair once and has no pair partial
    const bool fp = L.farlen_pair != nullptr && fa && fb && __ldg(L.farlen_pair + p * L.n + i) > 0;
    const size_t ea = static_cast<size_t>(zq) * m + 2 * i;
    const size_t tp = static_cast<size_t>(zq) * L.n + i;
    const float la = fa ? __ldg(L.lse_e + ea) : -INFINITY;
    const float lb = fb ? __ldg(L.lse_e + ea + 1) : -INFINITY;
    const float lp = fp ? __ldg(L.lse_p + tp) : -INFINITY;
    const float M = fmaxf(fmaxf(la, lb), lp);
    const float wa = fa ? expf(la - M) : 0.f;
    const float wb = fb ? expf(lb - M) : 0.f;
    const float wp = fp ? expf(lp - M) : 0.f;
    const float den = wa + wb - wp;
    const float inv = 1.f / den;
    const size_t col = static_cast<size_t>(part) * 8;
    Vec8<T> va{}, vb{}, vp{};
    if (fa) va.load(L.O_e, ea * L.d + col);
    if (fb) vb.load(L.O_e, (ea + 1) * L.d + col);
    if (fp) vp.load(L.O_p, tp * L.d + col);
    float o[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float x = 0.f;
      if (fa) x = fmaf(wa, va.get(e), x);
      if (fb) x = fmaf(wb, vb.get(e), x);
      if (fp) x = fmaf(-wp, vp.get(e), x);
      o[e] = x * inv;
    }
    Vec8<T> out;
    out.set_all(o);
    out.store(L.O_far, tp * L.d + col);
    if (part == 0) L.lse_far[tp] = M + logf(den);
  }
}

int grid_for(long long total) {
  const long long want = (total + 255) / 256;
  return static_cast<int>(want < 152LL * 16 ? (want > 0 ? want : 1) : 152LL * 16);
}

}  // namespace

cudaError_t launch_pair_ids(const int32_t* gid2, int P, int n, int K, int32_t* pair_gid, int* err,
                            cudaStream_t st) {
  const long long total = static_cast<long long>(P) * n;
  pair_ids_kernel<<<grid_for(total), 256, 0, st>>>(reinterpret_cast<const int2*>(gid2), total, K,
                                                   pair_gid, err);
  return cudaGetLastError();
}

cudaError_t launch_split_ids(const int32_t* gid2, int P, int n, int K, int32_t* vg, int* err, cudaStream_t st) {
  const long long total = static_cast<long long>(P) * n;
  split_ids_kernel<<<grid_for(total), 256, 0, st>>>(reinterpret_cast<const int2*>(gid2), total, K,
                                                    reinterpret_cast<int2*>(vg), err);
  return cudaGetLastError();
}

cudaError_t launch_far_any(const int32_t* farlen_entry, int P, int n, int32_t* far_any,
                           cudaStream_t st) {
  const long long total = static_cast<long long>(P) * n;
  far_any_kernel<<<grid_for(total), 256, 0, st>>>(reinterpret_cast<const int2*>(farlen_entry), total,
                                                  far_any);
  return cudaGetLastError();
}

cudaError_t launch_topk_merge(const MergeLaunch& L, int dtype, cudaStream_t st) {
  if (L.d % 8 != 0) return cudaErrorInvalidValue;
  const long long rows = static_cast<long long>(L.B) * L.H * L.n;
  const long long total = rows * (L.d / 8);
  if (dtype == FOCUS_BF16)
    topk_merge_kernel<__nv_bfloat16><<<grid_for(total), 256, 0, st>>>(L, rows);
  else
    topk_merge_kernel<float><<<grid_for(total), 256, 0, st>>>(L, rows);
  return cudaGetLastError();
}

}  // namespace focus
