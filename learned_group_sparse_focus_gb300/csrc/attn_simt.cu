// Focus attention for fp32 tensors on the CUDA cores (fp32 arithmetic).
//
// Same two-pass structure as the tensor-core path ("Why Attend to
// Everything? Focus is the Key", section 2.3; "Focus: Learning Which
// Attention Pairs Matter", section 3.3: the pattern splits into a local
// window part and an in-group causal part):
//   group pass  rows of one group in sorted order, keys = earlier members of
//               the group with j <= i - w; writes a normalised partial O and
//               its LSE at each row's item (token position, or the top-k
//               entry i * k + c of token i).
//   local pass  natural-order rows, keys j in [i - w + 1, i]; merges the
//               group partial (when the row has far keys) by log-sum-exp and
//               writes O.  The dense mode is the local pass with no partial:
//               with w = n every j <= i is kept (the comparator), with the
//               Focus window it is a standalone sliding-window call.
// A CTA holds 32 query rows, four threads per row (each owns d/4 of q and of
// the accumulator); keys stream through shared memory 32 at a time.
#include "common.cuh"
#include "kernels.h"

namespace focus {
namespace {

constexpr int kRows = 32;
constexpr int kKeys = 32;

__device__ __forceinline__ float fast_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D, int MODE>
__global__ void __launch_bounds__(128) attn_simt_kernel(AttnArgs a) {
  constexpr int DT = D / 4;
  __shared__ __align__(16) float Ks[kKeys][D];
  __shared__ __align__(16) float Vs[kKeys][D];
  __shared__ int key_pos[kKeys];

  const int tid = threadIdx.x;
  const int r = tid >> 2, part = tid & 3;
  const float* Q = static_cast<const float*>(a.Q);
  const float* Kg = static_cast<const float*>(a.Kg);
  const float* Vg = static_cast<const float*>(a.Vg);

  int b, h, kv, asg;
  int row_pos;            // token position of this thread's row (-1: none)
  int row_item = -1;      // group pass: the row's sorted item (O_far row)
  int lo, hi;             // kept key interval for this row (positions or slots)
  int key_begin, key_end; // key range the CTA walks
  const int32_t* perm_p = nullptr;
  int key0 = 0;
  int slot = -1;

  if (MODE == kModeGroup) {
    int L = blockIdx.x;
    const int sub = L % (kTileM / kRows);
    L /= kTileM / kRows;
    const int hpa = a.A == 1 ? a.H : a.H / a.H_kv;
    const int y = L % hpa;
    const int io = L / hpa;
    if (io >= *a.n_items) return;
    const focus_item_t it = a.items[a.order[io]];
    if (sub * kRows >= it.rows) return;
    b = it.b;
    asg = it.a;
    h = a.A == 1 ? y : it.a * (a.H / a.H_kv) + y;
    kv = (h * a.H_kv) / a.H;
    const int p = b * a.A + asg;
    perm_p = a.perm + static_cast<size_t>(p) * a.m;
    key0 = it.key0;
    const int rr = sub * kRows + r;
    const int last = min(it.rows, sub * kRows + kRows) - 1;
    key_begin = 0;
    key_end = a.farlen_slot[static_cast<size_t>(p) * a.m + it.row0 + last];
    if (rr < it.rows) {
      slot = it.row0 + rr;
      row_item = perm_p[slot];
      row_pos = row_item >> a.kshift;
      lo = 0;
      hi = a.farlen_slot[static_cast<size_t>(p) * a.m + slot] - 1;
    } else {
      row_pos = -1;
      lo = 1;
      hi = 0;
    }
  } else {
    int L = blockIdx.x;
    h = L % a.H;
    L /= a.H;
    const int nqt = (a.n + kRows - 1) / kRows;
    const int qt = nqt - 1 - (L % nqt);
    b = L / nqt;
    kv = (h * a.H_kv) / a.H;
    asg = a.A == 1 ? 0 : kv;
    const int i0 = qt * kRows;
    const int i = i0 + r;
    key_end = min(a.n, i0 + kRows);
    key_begin = max(0, i0 - a.w + 1);
    if (i < a.n) {
      row_pos = i;
      lo = i - a.w + 1;
      hi = i;
    } else {
      row_pos = -1;
      lo = 1;
      hi = 0;
    }
  }

  const size_t qrow = (static_cast<size_t>(b) * a.H + h) * a.n;
  const size_t kvrow = (static_cast<size_t>(b) * a.H_kv + kv) * a.n;

  float q[DT], acc[DT];
#pragma unroll
  for (int e = 0; e < DT; ++e) {
    q[e] = row_pos >= 0 ? Q[(qrow + row_pos) * D + part * DT + e] : 0.f;
    acc[e] = 0.f;
  }
  float m = -INFINITY, l = 0.f;

  for (int t0 = key_begin; t0 < key_end; t0 += kKeys) {
    __syncthreads();
    if (tid < kKeys) {
      const int t = t0 + tid;
      key_pos[tid] = t < key_end ? (MODE == kModeGroup ? perm_p[key0 + t] >> a.kshift : t) : -1;
    }
    __syncthreads();
    for (int e = tid; e < kKeys * D / 4; e += blockDim.x) {
      const int kk = e / (D / 4), c = (e % (D / 4)) * 4;
      const int pos = key_pos[kk];
      float4 kvv = make_float4(0.f, 0.f, 0.f, 0.f), vvv = kvv;
      if (pos >= 0) {
        kvv = *reinterpret_cast<const float4*>(Kg + (kvrow + pos) * D + c);
        vvv = *reinterpret_cast<const float4*>(Vg + (kvrow + pos) * D + c);
      }
      *reinterpret_cast<float4*>(&Ks[kk][c]) = kvv;
      *reinterpret_cast<float4*>(&Vs[kk][c]) = vvv;
    }
    __syncthreads();
    float s[kKeys];
    float mt = -INFINITY;
#pragma unroll
    for (int kk = 0; kk < kKeys; ++kk) {
      float d0 = 0.f;
#pragma unroll
      for (int e = 0; e < DT; ++e) d0 = fmaf(q[e], Ks[kk][part * DT + e], d0);
      d0 += __shfl_xor_sync(0xffffffffu, d0, 1);
      d0 += __shfl_xor_sync(0xffffffffu, d0, 2);
      const int t = t0 + kk;
      const bool keep = t >= lo && t <= hi && t < key_end;
      s[kk] = keep ? d0 * a.scale_log2 : -INFINITY;
      mt = fmaxf(mt, s[kk]);
    }
    const float mn = fmaxf(m, mt);
    if (mn == -INFINITY) continue;
    const float alpha = fast_ex2(m - mn);   // m = -inf -> 0
    l *= alpha;
#pragma unroll
    for (int e = 0; e < DT; ++e) acc[e] *= alpha;
#pragma unroll
    for (int kk = 0; kk < kKeys; ++kk) {
      const float pv = fast_ex2(s[kk] - mn);
      l += pv;
#pragma unroll
      for (int e = 0; e < DT; ++e) acc[e] = fmaf(pv, Vs[kk][part * DT + e], acc[e]);
    }
    m = mn;
  }

  if (row_pos < 0) return;
  const size_t orow = (qrow + row_pos) * D + part * DT;
  constexpr float kLn2 = 0.6931471805599453f;
  if (MODE == kModeGroup) {
    if (l > 0.f) {
      const size_t frow = (static_cast<size_t>(b) * a.H + h) * a.m + row_item;
      float* Of = static_cast<float*>(a.O_far) + frow * D + part * DT;
      const float inv = 1.f / l;
#pragma unroll
      for (int e = 0; e < DT; ++e) Of[e] = acc[e] * inv;
      if (part == 0) a.lse_far[frow] = (m + log2f(l)) * kLn2;
    }
    return;
  }
  float c1 = 1.f / l, c2 = 0.f;
  float lse2 = m + log2f(l);
  const float* Of = static_cast<const float*>(a.O_far);
  bool far = false;
  if (MODE == kModeLocal) {
    const int p = b * a.A + asg;
    far = a.farlen_tok[static_cast<size_t>(p) * a.n + row_pos] > 0;
    if (far) {
      const float lf2 = a.lse_far[qrow + row_pos] * 1.4426950408889634f;
      const float mm = fmaxf(lse2, lf2);
      const float e1 = fast_ex2(lse2 - mm), e2 = fast_ex2(lf2 - mm);
      const float den = e1 + e2;
      c1 = e1 / (l * den);
      c2 = e2 / den;
      lse2 = mm + log2f(den);
    }
  }
  float* O = static_cast<float*>(a.O);
#pragma unroll
  for (int e = 0; e < DT; ++e) {
    float v = acc[e] * c1;
    if (far) v = fmaf(Of[orow + e], c2, v);
    O[orow + e] = v;
  }
  if (a.lse && part == 0) a.lse[qrow + row_pos] = lse2 * kLn2;
}

template <int D>
cudaError_t launch_d(const AttnArgs& a, int mode, int max_items, cudaStream_t st) {
  if (mode == kModeGroup) {
    const int hpa = a.A == 1 ? a.H : a.H / a.H_kv;
    const long long grid = static_cast<long long>(max_items) * hpa * (kTileM / kRows);
    if (grid == 0) return cudaSuccess;
    attn_simt_kernel<D, kModeGroup><<<static_cast<unsigned>(grid), 128, 0, st>>>(a);
  } else {
    const long long grid = static_cast<long long>(a.B) * a.H * ((a.n + kRows - 1) / kRows);
    if (mode == kModeLocal)
      attn_simt_kernel<D, kModeLocal><<<static_cast<unsigned>(grid), 128, 0, st>>>(a);
    else
      attn_simt_kernel<D, kModeDense><<<static_cast<unsigned>(grid), 128, 0, st>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_simt_f32(const AttnArgs& a, int d, int mode, int max_items,
                                 cudaStream_t st) {
  if (d == 64) return launch_d<64>(a, mode, max_items, st);
  if (d == 128) return launch_d<128>(a, mode, max_items, st);
  return cudaErrorInvalidValue;
}

}  // namespace focus
