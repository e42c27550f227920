// The two-call comparator's combine step.
//
// "Why Attend to Everything? Focus is the Key", section 2.3 and "Focus:
// Learning Which Attention Pairs Matter", section 3.3 run Focus as two
// standard attention calls, a local-window one and an in-group causal one,
// whose results are combined afterwards; section 2.1 of the former: the
// softmax stays exact, i.e. the combine is a log-sum-exp merge.  The library's
// own path merges inside the local pass's epilogue; this kernel is the
// separate combine of the comparator that measures what that fusion saves.
//
// Per query row (zq, i) with far keys: O <- (e1 O + e2 O_far) / (e1 + e2),
// lse <- M + log(e1 + e2), e1 = exp(lse_loc - M), e2 = exp(lse_far - M),
// M = max(lse_loc, lse_far).  O is updated in place (each thread reads and
// writes only its own eight elements); rows without far keys keep the window
// call's O.
#include "common.cuh"
#include "kernels.h"

namespace focus {
namespace {

template <typename T>
struct Row8;
template <>
struct Row8<__nv_bfloat16> {
  static __device__ __forceinline__ void load(const void* base, size_t off, float* f) {
    const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + off);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      f[2 * e] = __uint_as_float(w[e] << 16);
      f[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
    }
  }
  static __device__ __forceinline__ void store(void* base, size_t off, const float* f) {
    uint4 u;
    u.x = pack_bf16x2(f[0], f[1]);
    u.y = pack_bf16x2(f[2], f[3]);
    u.z = pack_bf16x2(f[4], f[5]);
    u.w = pack_bf16x2(f[6], f[7]);
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + off) = u;
  }
};
template <>
struct Row8<float> {
  static __device__ __forceinline__ void load(const void* base, size_t off, float* f) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + off);
    const float4 a = p[0], b = p[1];
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  }
  static __device__ __forceinline__ void store(void* base, size_t off, const float* f) {
    float4* p = reinterpret_cast<float4*>(static_cast<float*>(base) + off);
    p[0] = make_float4(f[0], f[1], f[2], f[3]);
    p[1] = make_float4(f[4], f[5], f[6], f[7]);
  }
};

template <typename T>
__global__ void __launch_bounds__(256) lse_combine_kernel(CombineLaunch L, long long rows) {
  const int per_row = L.d / 8;
  const long long total = rows * per_row;
  for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t < total;
       t += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = t / per_row;
    const int part = static_cast<int>(t % per_row);
    const int i = static_cast<int>(row % L.n);
    const int zq = static_cast<int>(row / L.n);
    const int b = zq / L.H, h = zq % L.H;
    const int kv = (h * L.H_kv) / L.H;
    const size_t p = static_cast<size_t>(b) * L.A + (L.A == 1 ? 0 : kv);
    const float l1 = L.lse_loc[row];
    if (L.farlen_tok[p * L.n + i] <= 0) {
      if (part == 0 && L.lse_out) L.lse_out[row] = l1;
      continue;
    }
    const float l2 = L.lse_far[row];
    const float M = fmaxf(l1, l2);
    const float e1 = expf(l1 - M), e2 = expf(l2 - M);
    const float den = e1 + e2;
    const float c1 = e1 / den, c2 = e2 / den;
    const size_t off = static_cast<size_t>(row) * L.d + static_cast<size_t>(part) * 8;
    float o[8], f[8];
    Row8<T>::load(L.O, off, o);
    Row8<T>::load(L.O_far, off, f);
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = fmaf(c1, o[e], c2 * f[e]);
    Row8<T>::store(L.O, off, o);
    if (part == 0 && L.lse_out) L.lse_out[row] = M + logf(den);
  }
}

}  // namespace

cudaError_t launch_lse_combine(const CombineLaunch& L, int dtype, cudaStream_t st) {
  if (L.d % 8 != 0) return cudaErrorInvalidValue;
  const long long rows = static_cast<long long>(L.B) * L.H * L.n;
  const long long total = rows * (L.d / 8);
  const long long want = (total + 255) / 256;
  const int grid = static_cast<int>(want < 152LL * 16 ? (want > 0 ? want : 1) : 152LL * 16);
  if (dtype == FOCUS_BF16)
    lse_combine_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(L, rows);
  else
    lse_combine_kernel<float><<<grid, 256, 0, st>>>(L, rows);
  return cudaGetLastError();
}

}  // namespace focus
