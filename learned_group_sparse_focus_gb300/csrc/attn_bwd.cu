// Backward of Focus attention over the kept pairs (dQ, dK, dV), fp32
// arithmetic on the CUDA cores for fp32 and bf16 tensors.
//
// The gradient of exact softmax attention restricted to the kept pairs
// ("Why Attend to Everything? Focus is the Key", section 2.1: the softmax is
// the pretrained model's own, which is what lets a model be retrofitted and
// fine-tuned; "Focus: Learning Which Attention Pairs Matter", section 3.1).
// With P_ij = exp(scale q_i.k_j - LSE_i) on kept pairs (the forward's LSE),
// Delta_i = dO_i . O_i:
//   dV_j = sum_i P_ij dO_i,   dS_ij = P_ij (dO_i . v_j - Delta_i),
//   dQ_i = scale sum_j dS_ij k_j,   dK_j = scale sum_i dS_ij q_i,
// dK and dV summed over the query heads of a key/value head.
//
// The kept set splits as in the forward (window j > i - w, far j <= i - w in
// one group), and every kernel owns its output rows, so nothing is atomic:
//   delta    Delta_i per query row                                  warp/row
//   dq far   rows of a group-pass work item, keys = the group's earlier
//            members (the forward's items and farlen); dQ partial to ws
//   dq local natural rows, window keys; adds the far partial; writes dQ
//   dkv far  32 sorted slots per CTA as keys; queries = later members of the
//            key's group at positions >= j + w (a suffix of the group's
//            sorted run, found by binary search); dK/dV partials to ws
//   dkv local natural keys, queries i in [j, j + w - 1]; adds the far
//            partials; writes dK, dV
// A CTA holds 32 rows (queries or keys), four threads per row each owning d/4
// of the row's vectors; the other side streams through shared memory 32 rows
// at a time.
#include "common.cuh"
#include "kernels.h"

namespace focus {
namespace {

constexpr int kRows = 32;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float fast_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <typename T>
__device__ __forceinline__ float ld(const T* p, size_t i);
template <>
__device__ __forceinline__ float ld<float>(const float* p, size_t i) { return p[i]; }
template <>
__device__ __forceinline__ float ld<__nv_bfloat16>(const __nv_bfloat16* p, size_t i) {
  return __bfloat162float(p[i]);
}

template <typename T>
__device__ __forceinline__ void st(T* p, size_t i, float v);
template <>
__device__ __forceinline__ void st<float>(float* p, size_t i, float v) { p[i] = v; }
template <>
__device__ __forceinline__ void st<__nv_bfloat16>(__nv_bfloat16* p, size_t i, float v) {
  p[i] = __float2bfloat16_rn(v);
}

__device__ __forceinline__ float quad_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  return x;
}

// Delta_i = dO_i . O_i, one warp per (b, h, i) row.
template <typename T>
__global__ void __launch_bounds__(256) bwd_delta_kernel(BwdArgs a, long long rows) {
  const long long r = blockIdx.x * 8LL + warp_id();
  if (r >= rows) return;
  const T* O = static_cast<const T*>(a.O) + r * a.d;
  const T* dO = static_cast<const T*>(a.dO) + r * a.d;
  float s = 0.f;
  for (int e = lane_id(); e < a.d; e += 32) s = fmaf(ld(O, e), ld(dO, e), s);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane_id() == 0) a.delta[r] = s;
}

// ------------------------------------------------------------------ dQ ---
template <int D, typename T, int MODE>
__global__ void __launch_bounds__(128) bwd_dq_kernel(BwdArgs a) {
  constexpr int DT = D / 4;
  __shared__ __align__(16) float Ks[kRows][D];
  __shared__ __align__(16) float Vs[kRows][D];
  __shared__ int key_pos[kRows];
  const int tid = threadIdx.x;
  const int r = tid >> 2, part = tid & 3;
  const T* Q = static_cast<const T*>(a.Q);
  const T* Kg = static_cast<const T*>(a.K);
  const T* Vg = static_cast<const T*>(a.V);
  const T* dOg = static_cast<const T*>(a.dO);
  int b, h, kv, asg, row_pos, lo, hi, key_begin, key_end, key0 = 0;
  const int32_t* perm_p = nullptr;
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
    perm_p = a.perm + static_cast<size_t>(p) * a.n;
    key0 = it.key0;
    const int rr = sub * kRows + r;
    const int last = min(it.rows, sub * kRows + kRows) - 1;
    key_begin = 0;
    key_end = a.farlen_slot[static_cast<size_t>(p) * a.n + it.row0 + last];
    if (rr < it.rows) {
      const int slot = it.row0 + rr;
      row_pos = perm_p[slot];
      lo = 0;
      hi = a.farlen_slot[static_cast<size_t>(p) * a.n + slot] - 1;
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
  float q[DT], dov[DT], acc[DT];
  float lse2 = 0.f, dlt = 0.f;
#pragma unroll
  for (int e = 0; e < DT; ++e) {
    q[e] = row_pos >= 0 ? ld(Q, (qrow + row_pos) * D + part * DT + e) : 0.f;
    dov[e] = row_pos >= 0 ? ld(dOg, (qrow + row_pos) * D + part * DT + e) : 0.f;
    acc[e] = 0.f;
  }
  if (row_pos >= 0) {
    lse2 = a.lse[qrow + row_pos] * kLog2e;
    dlt = a.delta[qrow + row_pos];
  }
  for (int t0 = key_begin; t0 < key_end; t0 += kRows) {
    __syncthreads();
    if (tid < kRows) {
      const int t = t0 + tid;
      key_pos[tid] = t < key_end ? (MODE == kModeGroup ? perm_p[key0 + t] : t) : -1;
    }
    __syncthreads();
    for (int e = tid; e < kRows * D; e += blockDim.x) {
      const int kk = e / D, c = e % D;
      const int pos = key_pos[kk];
      Ks[kk][c] = pos >= 0 ? ld(Kg, (kvrow + pos) * D + c) : 0.f;
      Vs[kk][c] = pos >= 0 ? ld(Vg, (kvrow + pos) * D + c) : 0.f;
    }
    __syncthreads();
    for (int kk = 0; kk < kRows; ++kk) {
      float s = 0.f, dp = 0.f;
#pragma unroll
      for (int e = 0; e < DT; ++e) {
        s = fmaf(q[e], Ks[kk][part * DT + e], s);
        dp = fmaf(dov[e], Vs[kk][part * DT + e], dp);
      }
      s = quad_sum(s);
      dp = quad_sum(dp);
      const int t = t0 + kk;
      const bool keep = t >= lo && t <= hi && t < key_end;
      const float pr = keep ? fast_ex2(s * a.scale_log2 - lse2) : 0.f;
      const float ds = pr * (dp - dlt);
#pragma unroll
      for (int e = 0; e < DT; ++e) acc[e] = fmaf(ds, Ks[kk][part * DT + e], acc[e]);
    }
  }
  if (row_pos < 0) return;
  const size_t orow = (qrow + row_pos) * D + part * DT;
  if (MODE == kModeGroup) {
#pragma unroll
    for (int e = 0; e < DT; ++e) a.dq_far[orow + e] = acc[e] * a.scale;
    return;
  }
  const int p = b * a.A + asg;
  const bool far = a.farlen_tok[static_cast<size_t>(p) * a.n + row_pos] > 0;
  T* dQ = static_cast<T*>(a.dQ);
#pragma unroll
  for (int e = 0; e < DT; ++e) {
    float v = acc[e] * a.scale;
    if (far) v += a.dq_far[orow + e];
    st(dQ, orow + e, v);
  }
}

// ----------------------------------------------------------------- dK dV ---
template <int D, typename T, int MODE>
__global__ void __launch_bounds__(128) bwd_dkv_kernel(BwdArgs a) {
  constexpr int DT = D / 4;
  __shared__ __align__(16) float Qs[kRows][D];
  __shared__ __align__(16) float dOs[kRows][D];
  __shared__ float lse_s[kRows], dl_s[kRows];
  __shared__ int q_pos[kRows];
  __shared__ int range_lo, range_hi;
  const int tid = threadIdx.x;
  const int r = tid >> 2, part = tid & 3;
  const T* Q = static_cast<const T*>(a.Q);
  const T* Kg = static_cast<const T*>(a.K);
  const T* Vg = static_cast<const T*>(a.V);
  const T* dOg = static_cast<const T*>(a.dO);
  const int nkt = (a.n + kRows - 1) / kRows;
  int L = blockIdx.x;
  const int kt = L % nkt;
  L /= nkt;
  const int kv = L % a.H_kv;
  const int b = L / a.H_kv;
  const int asg = a.A == 1 ? 0 : kv;
  const int p = b * a.A + asg;
  const size_t kvrow = (static_cast<size_t>(b) * a.H_kv + kv) * a.n;
  const int32_t* perm_p = a.perm + static_cast<size_t>(p) * a.n;
  const int32_t* off_p = a.offsets + static_cast<size_t>(p) * (a.groups + 1);
  // this thread's key: natural position (local) or sorted slot (far)
  const int u = kt * kRows + r;
  int key_pos = -1, qlo = 1, qhi = 0;    // kept queries: [qlo, qhi] in the walked order
  if (u < a.n) {
    if (MODE == kModeGroup) {
      key_pos = perm_p[u];
      // group of slot u: largest g with off[g] <= u
      int glo = 0, ghi = a.groups;
      while (ghi - glo > 1) {
        const int mid = (glo + ghi) >> 1;
        if (off_p[mid] <= u) glo = mid; else ghi = mid;
      }
      const int gend = off_p[glo + 1];
      // first slot of the group at or after u whose position is >= key + w
      const int target = key_pos + a.w;
      int s0 = u + 1, s1 = gend;
      while (s0 < s1) {
        const int mid = (s0 + s1) >> 1;
        if (perm_p[mid] < target) s0 = mid + 1; else s1 = mid;
      }
      qlo = s0;
      qhi = gend - 1;
    } else {
      key_pos = u;
      qlo = u;
      qhi = min(a.n - 1, u + a.w - 1);
    }
  }
  if (tid == 0) {
    range_lo = 0x7fffffff;
    range_hi = -1;
  }
  __syncthreads();
  if (part == 0 && key_pos >= 0 && qlo <= qhi) {
    atomicMin(&range_lo, qlo);
    atomicMax(&range_hi, qhi);
  }
  __syncthreads();
  const int wlo = range_lo, whi = range_hi;
  float kr[DT], vr[DT], dk[DT], dv[DT];
#pragma unroll
  for (int e = 0; e < DT; ++e) {
    kr[e] = key_pos >= 0 ? ld(Kg, (kvrow + key_pos) * D + part * DT + e) : 0.f;
    vr[e] = key_pos >= 0 ? ld(Vg, (kvrow + key_pos) * D + part * DT + e) : 0.f;
    dk[e] = 0.f;
    dv[e] = 0.f;
  }
  const int hpk = a.H / a.H_kv;          // query heads per key/value head
  for (int hh = 0; hh < hpk && wlo <= whi; ++hh) {
    const int h = kv * hpk + hh;
    const size_t qrow = (static_cast<size_t>(b) * a.H + h) * a.n;
    for (int t0 = wlo; t0 <= whi; t0 += kRows) {
      __syncthreads();
      if (tid < kRows) {
        const int t = t0 + tid;
        const int pos = t <= whi ? (MODE == kModeGroup ? perm_p[t] : t) : -1;
        q_pos[tid] = pos;
        lse_s[tid] = pos >= 0 ? a.lse[qrow + pos] * kLog2e : 0.f;
        dl_s[tid] = pos >= 0 ? a.delta[qrow + pos] : 0.f;
      }
      __syncthreads();
      for (int e = tid; e < kRows * D; e += blockDim.x) {
        const int qq = e / D, c = e % D;
        const int pos = q_pos[qq];
        Qs[qq][c] = pos >= 0 ? ld(Q, (qrow + pos) * D + c) : 0.f;
        dOs[qq][c] = pos >= 0 ? ld(dOg, (qrow + pos) * D + c) : 0.f;
      }
      __syncthreads();
      for (int qq = 0; qq < kRows; ++qq) {
        float s = 0.f, dp = 0.f;
#pragma unroll
        for (int e = 0; e < DT; ++e) {
          s = fmaf(kr[e], Qs[qq][part * DT + e], s);
          dp = fmaf(vr[e], dOs[qq][part * DT + e], dp);
        }
        s = quad_sum(s);
        dp = quad_sum(dp);
        const int t = t0 + qq;
        const bool keep = t >= qlo && t <= qhi && q_pos[qq] >= 0;
        const float pr = keep ? fast_ex2(s * a.scale_log2 - lse_s[qq]) : 0.f;
        const float ds = pr * (dp - dl_s[qq]);
#pragma unroll
        for (int e = 0; e < DT; ++e) {
          dk[e] = fmaf(ds, Qs[qq][part * DT + e], dk[e]);
          dv[e] = fmaf(pr, dOs[qq][part * DT + e], dv[e]);
        }
      }
    }
  }
  if (key_pos < 0) return;
  const size_t orow = (kvrow + key_pos) * D + part * DT;
  if (MODE == kModeGroup) {
    // every key of the kv head is one sorted slot: all rows are written
#pragma unroll
    for (int e = 0; e < DT; ++e) {
      a.dk_far[orow + e] = dk[e] * a.scale;
      a.dv_far[orow + e] = dv[e];
    }
    return;
  }
  T* dK = static_cast<T*>(a.dK);
  T* dV = static_cast<T*>(a.dV);
#pragma unroll
  for (int e = 0; e < DT; ++e) {
    st(dK, orow + e, dk[e] * a.scale + a.dk_far[orow + e]);
    st(dV, orow + e, dv[e] + a.dv_far[orow + e]);
  }
}

template <int D, typename T>
cudaError_t launch_bwd_d(const BwdArgs& a, int max_items, cudaStream_t st) {
  const long long rows = static_cast<long long>(a.B) * a.H * a.n;
  bwd_delta_kernel<T><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, st>>>(a, rows);
  const int hpa = a.A == 1 ? a.H : a.H / a.H_kv;
  const long long g_items = static_cast<long long>(max_items) * hpa * (kTileM / kRows);
  if (g_items > 0) bwd_dq_kernel<D, T, kModeGroup><<<static_cast<unsigned>(g_items), 128, 0, st>>>(a);
  const long long q_tiles = static_cast<long long>(a.B) * a.H * ((a.n + kRows - 1) / kRows);
  bwd_dq_kernel<D, T, kModeLocal><<<static_cast<unsigned>(q_tiles), 128, 0, st>>>(a);
  const long long k_tiles = static_cast<long long>(a.B) * a.H_kv * ((a.n + kRows - 1) / kRows);
  bwd_dkv_kernel<D, T, kModeGroup><<<static_cast<unsigned>(k_tiles), 128, 0, st>>>(a);
  bwd_dkv_kernel<D, T, kModeLocal><<<static_cast<unsigned>(k_tiles), 128, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_delta(const BwdArgs& a, int dtype, cudaStream_t st) {
  const long long rows = static_cast<long long>(a.B) * a.H * a.n;
  const unsigned grid = static_cast<unsigned>((rows + 7) / 8);
  if (dtype == FOCUS_BF16)
    bwd_delta_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(a, rows);
  else
    bwd_delta_kernel<float><<<grid, 256, 0, st>>>(a, rows);
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd(const BwdArgs& a, int dtype, int max_items, cudaStream_t st) {
  if (dtype == FOCUS_BF16) {
    if (a.d == 64) return launch_bwd_d<64, __nv_bfloat16>(a, max_items, st);
    if (a.d == 128) return launch_bwd_d<128, __nv_bfloat16>(a, max_items, st);
  } else {
    if (a.d == 64) return launch_bwd_d<64, float>(a, max_items, st);
    if (a.d == 128) return launch_bwd_d<128, float>(a, max_items, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace focus
