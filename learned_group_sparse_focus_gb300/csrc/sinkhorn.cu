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
// The row step of round t and the column step of round t + 1 share one pass
// over S [P, n, K] (row-major, fp32): a row's potential u_i is known as soon as
// its K scores are in registers, so the same pass adds X_ik + u_i into running
// per-column (max, sum of exp) partials.  For K <= 256, K % 4 == 0 each round
// is one launch of the pass kernel: one read of S, in base 2 with the hardware
// exp2: eight lanes per row with float4 loads, 8-lane shuffle LSE -> u_i,
// then the next round's column partials (combined across the warp by
// shuffles, across the block's warps in shared memory, and across the blocks
// of a problem by the last of them to finish, which writes the next v), or in
// the last round G (may alias S: each lane reads its elements before writing
// them, and rows are disjoint).  Round 1's column step is a pass with u = 0
// and no row step, so T rounds are T + 1 reads of S, one write of G and T + 1
// launches.
// Other K take three launches and two reads of S per round: colpart (per row
// chunk and column, running max and sum of exp), colfin, and the row kernel
// (LR lanes per row) that writes u, and G in the last round.  Memory-bound.
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

__device__ __forceinline__ float ex2a(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Running (max, sum of 2^(y - max)) of a column in base 2.  The max moves only
// when a value exceeds it by more than 16, so the common step is one exp2 and
// one add (a sum of at most 2^24 terms below 2^16 cannot overflow).
__device__ __forceinline__ void lse2_push(float& m, float& s, float y) {
  if (y > m + 16.f) {
    s = s * ex2a(m - y) + 1.f;
    m = y;
  } else if (m != -INFINITY) {
    s += ex2a(y - m);
  }
}

__device__ __forceinline__ void lse2_join(float& m, float& s, float m2, float s2) {
  if (s2 == 0.f) return;
  if (s == 0.f) {
    m = m2;
    s = s2;
    return;
  }
  if (m2 > m) {
    s = s * ex2a(m - m2) + s2;
    m = m2;
  } else {
    s += s2 * ex2a(m2 - m);
  }
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

// warp-uniform bounded wait (every lane waits; the outcome is shared)
__device__ __forceinline__ bool all_wait(uint64_t* bar, uint32_t parity, volatile int* abort, int* err) {
  const bool ok = mbar_wait(bar, parity, abort, err);
  return __all_sync(0xffffffffu, ok);
}

// one arrival per warp, after every lane is done with the stage
__device__ __forceinline__ void warp_release(uint64_t* bar, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

constexpr int kPassStages = 6;
constexpr int kPassStageBytes = 32768;
constexpr int kPassSmem = kPassStages * kPassStageBytes + 256;
// compute warps per block (plus one load warp): 16 up to 64 columns, 8 above
// (where registers per thread would not allow 16)
__host__ __device__ constexpr int pass_warps(int NV) { return NV <= 2 ? 16 : 8; }

// Rows per 32 KB stage for K columns (a multiple of 32 rows).
__host__ __device__ inline int pass_stage_rows(int K) { return (kPassStageBytes / (4 * K)) / 32 * 32; }

// One pass over rows [r0, r1) of problem p (K % 4 == 0, K <= 256), base 2:
// X2 = S log2(e) / tau, v2 = v log2(e).  kMode 0: the row step
// u2_i = -log2 sum_k 2^(X2_ik + v2_k), then the next round's column partials
// of X2 + u2; 1: the last round's G_ik = 2^(X2_ik + u2_i + v2_k); 2: round 1's
// column partials of X2 (u = 0, no row step).  The chunk is contiguous in S:
// warp 8 streams it through a ring of six 32 KB stages with bulk copies, and
// the compute warps take eight lanes per row, lane lr holding columns
// 4 lr + 32 j .. + 3 (j < NV), four rows per warp per sweep, two sweeps at a
// time.  In modes 0 and 2 the last block of a problem to finish (a ticket per
// problem) combines every chunk's partials into the next v.
template <int NV, int kMode>
__global__ void __launch_bounds__(32 * (pass_warps(NV) + 1), 1)
    sinkhorn_pass_kernel(SinkhornLaunch L, int rows_per_chunk) {
  constexpr int kWarps = pass_warps(NV), kSweep = 4 * kWarps;
  constexpr float kLog2e = 1.4426950408889634f, kLn2 = 0.6931471805599453f;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float2 red[kMode == 1 ? 1 : kWarps][kMode == 1 ? 1 : NV * 32];
  __shared__ int last;
  __shared__ int abort_flag;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kPassStages * kPassStageBytes);
  uint64_t* empty = full + kPassStages;
  volatile int* abort = &abort_flag;
  const int p = blockIdx.y, chunk = blockIdx.x;
  const int K = L.K, n = L.n;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = chunk * rows_per_chunk, r1 = min(n, r0 + rows_per_chunk);
  const int SR = pass_stage_rows(K);
  const int ns = r1 > r0 ? (r1 - r0 + SR - 1) / SR : 0;
  if (threadIdx.x == 0) {
    for (int t = 0; t < kPassStages; ++t) {
      mbar_init(&full[t], 1);
      mbar_init(&empty[t], kWarps);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const float* S = L.S + static_cast<size_t>(p) * n * K;

  if (warp == kWarps) {
    // ------------------------------------------------------------ loads ---
    if (lane == 0) {
      int t = 0;
      for (; t < ns; ++t) {
        const int slot = t % kPassStages, use = t / kPassStages;
        if (use > 0 && !mbar_wait_nap(&empty[slot], (use - 1) & 1, abort, L.err)) break;
        const int rows = min(SR, r1 - r0 - t * SR);
        const uint32_t bytes = static_cast<uint32_t>(rows) * K * 4;
        mbar_expect_tx(&full[slot], bytes);
        bulk_load(smem + slot * kPassStageBytes, S + static_cast<size_t>(r0 + t * SR) * K, bytes, &full[slot]);
      }
      // copies in flight must land before the block exits
      for (int j = max(0, t - kPassStages); j < t; ++j) {
        const unsigned long long t0 = global_ns();
        while (!mbar_try_wait(&full[j % kPassStages], (j / kPassStages) & 1) &&
               global_ns() - t0 < kWaitTimeoutNs) {}
      }
    }
  } else {
    // ---------------------------------------------------------- compute ---
    const int lr = lane & 7, g = lane >> 3;
    const float c = L.inv_tau * kLog2e;
    float v2[NV][4], cm[NV][4], cs[NV][4];
    bool has[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int k0 = 4 * lr + 32 * j;
      has[j] = k0 < K;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v2[j][e] = (kMode != 2 && has[j]) ? L.v[static_cast<size_t>(p) * K + k0 + e] * kLog2e : 0.f;
        cm[j][e] = -INFINITY;
        cs[j][e] = 0.f;
      }
    }
    for (int t = 0; t < ns; ++t) {
      const int slot = t % kPassStages;
      if (!all_wait(&full[slot], (t / kPassStages) & 1, abort, L.err)) break;
      const float* st = reinterpret_cast<const float*>(smem + slot * kPassStageBytes);
      const int rows = min(SR, r1 - r0 - t * SR);
      // two sweeps of kSweep rows per step; rows past the stage count as -inf
      for (int sw = 0; sw < rows; sw += 2 * kSweep) {
        float xs[2][NV][4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int rr = sw + kSweep * h + warp * 4 + g;
#pragma unroll
          for (int j = 0; j < NV; ++j) {
            float4 x4 = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            if (rr < rows && has[j]) x4 = *reinterpret_cast<const float4*>(st + static_cast<size_t>(rr) * K + 4 * lr + 32 * j);
            xs[h][j][0] = x4.x * c;
            xs[h][j][1] = x4.y * c;
            xs[h][j][2] = x4.z * c;
            xs[h][j][3] = x4.w * c;
          }
        }
        if (kMode == 2) {
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int j = 0; j < NV; ++j)
#pragma unroll
              for (int e = 0; e < 4; ++e) lse2_push(cm[j][e], cs[j][e], xs[h][j][e]);
          continue;
        }
        // row step: e_k = 2^(X2 + v2 - max), G_ik = e_k / sum_k e_k
        float m[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int j = 0; j < NV; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              xs[h][j][e] += v2[j][e];
              m[h] = fmaxf(m[h], xs[h][j][e]);
            }
#pragma unroll
        for (int o = 1; o < 8; o <<= 1)
#pragma unroll
          for (int h = 0; h < 2; ++h) m[h] = fmaxf(m[h], __shfl_xor_sync(0xffffffffu, m[h], o));
        float sum[2] = {0.f, 0.f};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          // an all -inf row (or a row past the stage) has no mass: it adds nothing
          const float mr = m[h] == -INFINITY ? 0.f : m[h];
#pragma unroll
          for (int j = 0; j < NV; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              xs[h][j][e] = ex2a(xs[h][j][e] - mr);
              sum[h] += xs[h][j][e];
            }
        }
#pragma unroll
        for (int o = 1; o < 8; o <<= 1)
#pragma unroll
          for (int h = 0; h < 2; ++h) sum[h] += __shfl_xor_sync(0xffffffffu, sum[h], o);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float rs = sum[h] > 0.f ? __fdividef(1.f, sum[h]) : 0.f;
          const int rr = sw + kSweep * h + warp * 4 + g;
          if (kMode == 1) {
            if (rr < rows) {
              float* G = L.G + (static_cast<size_t>(p) * n + r0 + t * SR + rr) * K;
#pragma unroll
              for (int j = 0; j < NV; ++j)
                if (has[j])
                  *reinterpret_cast<float4*>(G + 4 * lr + 32 * j) =
                      make_float4(xs[h][j][0] * rs, xs[h][j][1] * rs, xs[h][j][2] * rs, xs[h][j][3] * rs);
            }
          } else {
            // next round's column partials: after the row step every G_ik <= 1
            // and each column's total is at least 1/K of its mass before it,
            // so the plain sum of G_ik (reference -v2_k) neither overflows nor
            // loses the column
#pragma unroll
            for (int j = 0; j < NV; ++j)
#pragma unroll
              for (int e = 0; e < 4; ++e) cs[j][e] = fmaf(xs[h][j][e], rs, cs[j][e]);
          }
        }
      }
      warp_release(&empty[slot], lane);
    }
    if (kMode == 0) {
#pragma unroll
      for (int j = 0; j < NV; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) cm[j][e] = cs[j][e] > 0.f ? -v2[j][e] : -INFINITY;
    }
    if (kMode != 1) {
      // the four row groups of a warp hold partials of the same columns
#pragma unroll
      for (int o = 8; o < 32; o <<= 1)
#pragma unroll
        for (int j = 0; j < NV; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float m2 = __shfl_xor_sync(0xffffffffu, cm[j][e], o);
            const float s2 = __shfl_xor_sync(0xffffffffu, cs[j][e], o);
            lse2_join(cm[j][e], cs[j][e], m2, s2);
          }
      if (g == 0) {
#pragma unroll
        for (int j = 0; j < NV; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) red[warp][4 * lr + 32 * j + e] = make_float2(cm[j][e], cs[j][e]);
      }
    }
  }
  __syncwarp();
  __syncthreads();
  if (kMode == 1 || *abort) return;
  float2* part = L.part + static_cast<size_t>(p) * gridDim.x * K;
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    float m = red[0][k].x, sm = red[0][k].y;
    for (int w = 1; w < kWarps; ++w) lse2_join(m, sm, red[w][k].x, red[w][k].y);
    part[static_cast<size_t>(chunk) * K + k] = make_float2(sm > 0.f ? m * kLn2 : -INFINITY, sm);
  }
  // the last block of problem p to get here turns all partials into v
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(L.ticket + p, 1) == static_cast<int>(gridDim.x) - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  const int nc = gridDim.x;
  const int per = (kWarps * 32) / K;       // threads per column (>= 1 for K <= 256)
  static_assert(kWarps * NV * 32 >= kWarps * 32, "red holds a value per compute thread");
  const int k = threadIdx.x % K, q = threadIdx.x / K;
  float m = -INFINITY, sm = 0.f;
  if (threadIdx.x < kWarps * 32 && q < per) {
    // sixteen independent loads in flight per step
    constexpr int kB = 16;
    for (int ch0 = q; ch0 < nc; ch0 += kB * per) {
      float2 tv[kB];
#pragma unroll
      for (int b = 0; b < kB; ++b) {
        const int ch = ch0 + b * per;
        tv[b] = ch < nc ? __ldcg(part + static_cast<size_t>(ch) * K + k) : make_float2(-INFINITY, 0.f);
      }
#pragma unroll
      for (int b = 0; b < kB; ++b) lse_join(m, sm, tv[b].x, tv[b].y);
    }
  }
  __syncthreads();                         // red is reused
  float2* red2 = &red[0][0];               // kWarps * NV * 32 >= kWarps * 32 entries
  if (threadIdx.x < kWarps * 32) red2[threadIdx.x] = make_float2(m, sm);
  __syncthreads();
  if (threadIdx.x < K) {
    m = red2[threadIdx.x].x;
    sm = red2[threadIdx.x].y;
    for (int w = 1; w < per; ++w) lse_join(m, sm, red2[w * K + threadIdx.x].x, red2[w * K + threadIdx.x].y);
    const float target = logf(static_cast<float>(n) / static_cast<float>(K));
    // an all -inf column has no mass to scale: its potential stays 0
    L.v[static_cast<size_t>(p) * K + threadIdx.x] = sm > 0.f ? target - (m + logf(sm)) : 0.f;
  }
  if (threadIdx.x == 0) L.ticket[p] = 0;   // ready for the next pass
}

template <int NV>
void launch_pass(const SinkhornLaunch& L, int rpc, int chunks, int mode, cudaStream_t st) {
  const dim3 grid(chunks, L.P);
  constexpr int threads = 32 * (pass_warps(NV) + 1);
  if (mode == 0) sinkhorn_pass_kernel<NV, 0><<<grid, threads, kPassSmem, st>>>(L, rpc);
  else if (mode == 1) sinkhorn_pass_kernel<NV, 1><<<grid, threads, kPassSmem, st>>>(L, rpc);
  else sinkhorn_pass_kernel<NV, 2><<<grid, threads, kPassSmem, st>>>(L, rpc);
}

void launch_pass_k(const SinkhornLaunch& L, int rpc, int chunks, int mode, cudaStream_t st) {
  if (L.K <= 32) launch_pass<1>(L, rpc, chunks, mode, st);
  else if (L.K <= 64) launch_pass<2>(L, rpc, chunks, mode, st);
  else if (L.K <= 128) launch_pass<4>(L, rpc, chunks, mode, st);
  else launch_pass<8>(L, rpc, chunks, mode, st);
}

template <int NV>
cudaError_t set_pass_smem() {
  cudaError_t e = cudaFuncSetAttribute(sinkhorn_pass_kernel<NV, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPassSmem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(sinkhorn_pass_kernel<NV, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPassSmem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(sinkhorn_pass_kernel<NV, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPassSmem);
  return e;
}

}  // namespace

cudaError_t setup_sinkhorn_kernels() {
  cudaError_t e = set_pass_smem<1>();
  if (e == cudaSuccess) e = set_pass_smem<2>();
  if (e == cudaSuccess) e = set_pass_smem<4>();
  if (e == cudaSuccess) e = set_pass_smem<8>();
  return e;
}

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
  if (L.K <= 256 && L.K % 4 == 0) {
    // one block per SM over all problems (each streams a contiguous chunk),
    // no more chunks than the partial buffer holds
    const int want = (L.num_sms + L.P - 1) / L.P;
    const int fchunks = chunks < want ? chunks : want;
    const int frpc = (L.n + fchunks - 1) / fchunks;
    const int fc = (L.n + frpc - 1) / frpc;
    e = cudaMemsetAsync(L.ticket, 0, static_cast<size_t>(L.P) * sizeof(int), st);
    if (e == cudaSuccess) launch_pass_k(L, frpc, fc, 2, st);
    for (int t = 0; t < iters && e == cudaSuccess; ++t) {
      launch_pass_k(L, frpc, fc, t == iters - 1 ? 1 : 0, st);
      e = cudaGetLastError();
    }
    return e;
  }
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
