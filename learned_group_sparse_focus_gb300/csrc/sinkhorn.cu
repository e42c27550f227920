// Sinkhorn soft assignment, forward (the training-time assignment of Focus).
//
// "Focus: Learning Which Attention Pairs Matter", sections 2.1 and 2.3; "Why
// Attend to Everything? Focus is the Key", section 2.2: tokens are assigned
// softly to the K groups, and Sinkhorn normalisation forces the n x K
// assignment matrix to be doubly stochastic, so every group receives an
// equal share of the tokens.  For each problem (b, a), X = S / tau:
//   G = diag(e^u) exp(X) diag(e^v),  rows of G sum to 1, columns to n / K,
// reached by T rounds of Sinkhorn-Knopp scaling, each round first the
// columns, then the rows, kept here in the log domain (potentials u, v):
//   v_k = log(n / K) - LSE_i (X_ik + u_i),   u_i = -LSE_k (X_ik + v_k),
// starting from u = 0, and G_ik = exp(X_ik + u_i + v_k) after the last round.
//
// Per round, three launches over S [P, n, K] (row-major, fp32):
//   colpart  per (row chunk, column): running max and sum of exp over the
//            chunk's rows (grid: chunks x P; consecutive threads read
//            consecutive columns of a row)
//   colfin   per column: combine the chunk partials -> v
//            (grid: K/32 x P; 32 columns x 32 chunk lanes per block)
//   row      LR lanes per row (8 for K <= 128, else the whole warp): LSE
//            over the K columns with v from shared memory -> u; the last
//            round also writes G (may alias S: each lane reads its elements
//            before writing them, and rows are disjoint)
// Memory-bound: each round streams S twice.
#include "common.cuh"
#include "kernels.h"

namespace focus {
namespace {

__device__ __forceinline__ void lse_push(float& m, float& s, float x) {
  if (x == -INFINITY) return;
  if (x > m) {
    s = s * expf(m - x) + 1.f;
    m = x;
  } else {
    s += expf(x - m);
  }
}

__device__ __forceinline__ void lse_join(float& m, float& s, float m2, float s2) {
  if (s2 == 0.f) return;
  if (s == 0.f) {
    m = m2;
    s = s2;
    return;
  }
  if (m2 > m) {
    s = s * expf(m - m2) + s2;
    m = m2;
  } else {
    s += s2 * expf(m2 - m);
  }
}

__global__ void __launch_bounds__(256) sinkhorn_colpart_kernel(SinkhornLaunch L, int rows_per_chunk) {
  extern __shared__ float2 red[];      // [lanes][kc]
  const int p = blockIdx.y, chunk = blockIdx.x;
  const int K = L.K, n = L.n;
  const int kc = K < 256 ? K : 256;
  const int lanes = 256 / kc;
  const int t = threadIdx.x;
  const int kl = t % kc, lane = t / kc;
  const int r0 = chunk * rows_per_chunk, r1 = min(n, r0 + rows_per_chunk);
  const float* S = L.S + static_cast<size_t>(p) * n * K;
  const float* u = L.u + static_cast<size_t>(p) * n;
  for (int k0 = 0; k0 < K; k0 += kc) {
    const int k = k0 + kl;
    float m = -INFINITY, s = 0.f;
    if (lane < lanes && k < K) {
      int i = r0 + lane;
      // four rows' loads in flight before their exps
      for (; i + 3 * lanes < r1; i += 4 * lanes) {
        const float x0 = __ldg(S + static_cast<size_t>(i) * K + k) * L.inv_tau + u[i];
        const float x1 = __ldg(S + static_cast<size_t>(i + lanes) * K + k) * L.inv_tau + u[i + lanes];
        const float x2 = __ldg(S + static_cast<size_t>(i + 2 * lanes) * K + k) * L.inv_tau + u[i + 2 * lanes];
        const float x3 = __ldg(S + static_cast<size_t>(i + 3 * lanes) * K + k) * L.inv_tau + u[i + 3 * lanes];
        lse_push(m, s, x0);
        lse_push(m, s, x1);
        lse_push(m, s, x2);
        lse_push(m, s, x3);
      }
      for (; i < r1; i += lanes) lse_push(m, s, __ldg(S + static_cast<size_t>(i) * K + k) * L.inv_tau + u[i]);
    }
    __syncthreads();
    if (lane < lanes) red[lane * kc + kl] = make_float2(m, s);
    __syncthreads();
    if (lane == 0 && k < K) {
      for (int l = 1; l < lanes; ++l) lse_join(m, s, red[l * kc + kl].x, red[l * kc + kl].y);
      L.part[(static_cast<size_t>(p) * gridDim.x + chunk) * K + k] = make_float2(m, s);
    }
  }
}

__global__ void __launch_bounds__(1024) sinkhorn_colfin_kernel(SinkhornLaunch L, int chunks) {
  __shared__ float2 red[32][33];
  const int p = blockIdx.y;
  const int k = blockIdx.x * 32 + threadIdx.x;
  const int y = threadIdx.y;
  float m = -INFINITY, s = 0.f;
  if (k < L.K) {
    const float2* part = L.part + static_cast<size_t>(p) * chunks * L.K + k;
    int c = y;
    // four independent loads in flight per step
    for (; c + 96 < chunks; c += 128) {
      const float2 q0 = part[static_cast<size_t>(c) * L.K];
      const float2 q1 = part[static_cast<size_t>(c + 32) * L.K];
      const float2 q2 = part[static_cast<size_t>(c + 64) * L.K];
      const float2 q3 = part[static_cast<size_t>(c + 96) * L.K];
      lse_join(m, s, q0.x, q0.y);
      lse_join(m, s, q1.x, q1.y);
      lse_join(m, s, q2.x, q2.y);
      lse_join(m, s, q3.x, q3.y);
    }
    for (; c < chunks; c += 32) {
      const float2 q = part[static_cast<size_t>(c) * L.K];
      lse_join(m, s, q.x, q.y);
    }
  }
  red[y][threadIdx.x] = make_float2(m, s);
  __syncthreads();
  if (y == 0 && k < L.K) {
    for (int l = 1; l < 32; ++l) lse_join(m, s, red[l][threadIdx.x].x, red[l][threadIdx.x].y);
    const float target = logf(static_cast<float>(L.n) / static_cast<float>(L.K));
    // an all -inf column has no mass to scale: leave its potential at 0
    L.v[static_cast<size_t>(p) * L.K + k] = s > 0.f ? target - (m + logf(s)) : 0.f;
  }
}

template <int LR>
__global__ void __launch_bounds__(256) sinkhorn_row_kernel(SinkhornLaunch L, int write_g) {
  extern __shared__ float vs[];        // [K]
  constexpr int kRowsPerBlock = 256 / LR;
  const int p = blockIdx.y;
  const int K = L.K;
  for (int k = threadIdx.x; k < K; k += blockDim.x) vs[k] = L.v[static_cast<size_t>(p) * K + k];
  __syncthreads();
  const int lr = threadIdx.x % LR;
  const int i = blockIdx.x * kRowsPerBlock + threadIdx.x / LR;
  // rows past n still join the shuffles (LR < 32 shares a warp between rows)
  const bool valid = i < L.n;
  const size_t row = (static_cast<size_t>(p) * L.n + (valid ? i : 0)) * K;
  const float* S = L.S + row;
  float m = -INFINITY, s = 0.f;
  if (valid)
    for (int k = lr; k < K; k += LR) lse_push(m, s, S[k] * L.inv_tau + vs[k]);
#pragma unroll
  for (int o = LR / 2; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    lse_join(m, s, m2, s2);
  }
  if (!valid) return;
  const float ui = s > 0.f ? -(m + logf(s)) : 0.f;
  if (lr == 0) L.u[static_cast<size_t>(p) * L.n + i] = ui;
  if (write_g) {
    float* G = L.G + row;
    for (int k = lr; k < K; k += LR) G[k] = expf(S[k] * L.inv_tau + ui + vs[k]);
  }
}

}  // namespace

int sinkhorn_rows_per_chunk(int n) {
  // at most 2048 chunks per problem, at least 128 rows each
  const int r = (n + 2047) / 2048;
  return r < 128 ? 128 : r;
}

cudaError_t launch_sinkhorn(const SinkhornLaunch& L, int iters, cudaStream_t st) {
  const int rpc = sinkhorn_rows_per_chunk(L.n);
  const int chunks = (L.n + rpc - 1) / rpc;
  const int kc = L.K < 256 ? L.K : 256;
  const size_t sm_part = static_cast<size_t>(256 / kc) * kc * sizeof(float2);
  const size_t sm_row = static_cast<size_t>(L.K) * sizeof(float);
  // u = 0 before the first round
  cudaError_t e = cudaMemsetAsync(L.u, 0, static_cast<size_t>(L.P) * L.n * sizeof(float), st);
  for (int t = 0; t < iters && e == cudaSuccess; ++t) {
    sinkhorn_colpart_kernel<<<dim3(chunks, L.P), 256, sm_part, st>>>(L, rpc);
    sinkhorn_colfin_kernel<<<dim3((L.K + 31) / 32, L.P), dim3(32, 32), 0, st>>>(L, chunks);
    if (L.K <= 128)
      sinkhorn_row_kernel<8><<<dim3((L.n + 31) / 32, L.P), 256, sm_row, st>>>(L, t == iters - 1);
    else
      sinkhorn_row_kernel<32><<<dim3((L.n + 7) / 8, L.P), 256, sm_row, st>>>(L, t == iters - 1);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace focus
