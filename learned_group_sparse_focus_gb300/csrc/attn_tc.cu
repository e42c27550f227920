// Focus attention on the tcgen05 tensor cores (bf16 in, fp32 accumulate).
//
// "Focus: Learning Which Attention Pairs Matter", section 2.1: local window
// pairs at full resolution, far pairs only inside a group; section 2.2: far
// pairs of different groups are skipped outright; section 3.3 and "Why Attend
// to Everything? Focus is the Key", section 2.3: the pattern splits into a
// local-window attention and an in-group causal attention whose softmaxes
// combine exactly ("Why Attend to Everything?", section 2.1).
//
// One kernel, three modes, one CTA per 128-row query tile:
//   group  rows = one work item (<= 128 sorted slots of one group), keys =
//          the group's earlier members at or before i - w (slot < farlen of
//          the row), read from K/V pre-permuted into sorted order so every
//          key tile is a dense TMA box.  Writes the normalised partial O and
//          its LSE at each row's token position.
//   local  rows = 128 consecutive tokens, keys j in [i - w + 1, i]; merges the
//          group partial by log-sum-exp when the row has far keys; writes O.
//   dense  rows = 128 consecutive tokens, every j <= i (the comparator).
//
// Warp roles (192 threads):
//   warp 0       TMA producer: K and V tiles, 2-stage rings
//   warp 1       TMEM owner and MMA issuer: S = Q K^T (SS, both K-major),
//                O += P V (TS: P from TMEM, V MN-major in shared memory)
//   warps 2..5   softmax: one query row per thread.  Reads S from TMEM,
//                applies the keep rule to boundary tiles, online max/sum in
//                fp32 (exp2 domain), writes P as bf16 into TMEM, rescales O in
//                TMEM only when the running max grows by more than 2^8, and
//                runs the epilogue.
// TMEM: S double buffer (2 x 128 cols), O (d cols), P double buffer (2 x 64).
// Every wait is bounded; on timeout the CTA raises an error bit, drains its
// copies, frees TMEM and exits.
#include "common.cuh"
#include "kernels.h"

namespace focus {
namespace {

constexpr int kBN = 128;
constexpr float kRescaleThreshold = 8.0f;   // log2 units

template <int D>
struct AttnCfg {
  static constexpr int kChunk = 128 * 128;            // 128 rows x 128 B
  static constexpr int kTile = 128 * D * 2;           // one Q/K/V tile
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTile;               // 2 stages
  static constexpr int kV = kK + 2 * kTile;           // 2 stages
  static constexpr int kBar = kV + 2 * kTile;
  // at least ~116 KB so that one CTA owns an SM (and its whole TMEM)
  static constexpr int kSmemRaw = kBar + 256 + 1024;
  static constexpr int kSmem = kSmemRaw < 118 * 1024 ? 118 * 1024 : kSmemRaw;
  static constexpr uint32_t kS0 = 0, kO = 256, kP0 = 256 + D;
  static constexpr uint32_t kTmemCols = 512;
};

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// warp-uniform bounded wait (every lane waits; the verdict is shared)
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          int* err) {
  const bool ok = mbar_wait(bar, parity, abort, err);
  return __all_sync(0xffffffffu, ok);
}

template <int D, int MODE>
__global__ void __launch_bounds__(192, 1) attn_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                         const __grid_constant__ CUtensorMap tm_v,
                                                         const AttnArgs a) {
  using Cfg = AttnCfg<D>;
  constexpr int kChunks = D / 64;

  // ---------------------------------------------------- work (uniform) ---
  int b, h, kv, asg, nt, ybase, row_base, nrows;
  int key0 = 0;
  if (MODE == kModeGroup) {
    const int hpa = a.A == 1 ? a.H : a.H / a.H_kv;
    const int y = blockIdx.x % hpa;
    const int io = blockIdx.x / hpa;
    if (io >= *a.n_items) return;
    const focus_item_t it = a.items[a.order[io]];
    b = it.b;
    asg = it.a;
    h = a.A == 1 ? y : it.a * (a.H / a.H_kv) + y;
    kv = (h * a.H_kv) / a.H;
    nt = (it.keys + kBN - 1) / kBN;
    ybase = it.key0;
    key0 = it.key0;
    row_base = it.row0;
    nrows = it.rows;
  } else {
    int L = blockIdx.x;
    h = L % a.H;
    L /= a.H;
    const int nqt = (a.n + kTileM - 1) / kTileM;
    const int qt = nqt - 1 - (L % nqt);          // longest tiles first
    b = L / nqt;
    kv = (h * a.H_kv) / a.H;
    asg = a.A == 1 ? 0 : kv;
    row_base = qt * kTileM;
    nrows = min(kTileM, a.n - row_base);
    const int jt0 = MODE == kModeDense ? 0 : max(0, row_base - a.w + 1) / kBN;
    const int jt1 = (row_base + nrows - 1) / kBN;
    nt = jt1 - jt0 + 1;
    ybase = jt0 * kBN;
  }
  (void)key0;
  const int prob = b * a.A + asg;
  const int zkv = b * a.H_kv + kv;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + Cfg::kQ;
  uint8_t* sK = smem + Cfg::kK;
  uint8_t* sV = smem + Cfg::kV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kBar);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = bars + 3;
  uint64_t* v_full = bars + 5;
  uint64_t* v_empty = bars + 7;
  uint64_t* s_full = bars + 9;
  uint64_t* p_ready = bars + 11;
  uint64_t* o_done = bars + 13;    // one phase per PV product (waited only while
                                   // at most one phase behind: see the rescale)
  uint64_t* o_final = bars + 14;   // single phase: every PV product is done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 15);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    mbar_init(q_full, 128);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
      mbar_init(&s_full[s], 1);
      mbar_init(&p_ready[s], 128);
    }
    mbar_init(o_done, 1);
    mbar_init(o_final, 1);
    *abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  if (warp == 1) tmem_alloc(tmem_slot, Cfg::kTmemCols);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------- producer ---
    if (lane == 0) {
      int k_issued = 0, v_issued = 0;
      for (int t = 0; t < nt; ++t) {
        const int st = t & 1, u = t >> 1;
        const int y = ybase + t * kBN;
        if (u > 0 && !mbar_wait(&k_empty[st], (u - 1) & 1, abort, a.err)) break;
        mbar_expect_tx(&k_full[st], Cfg::kTile);
#pragma unroll
        for (int c = 0; c < kChunks; ++c)
          tma_load_3d(sK + st * Cfg::kTile + c * Cfg::kChunk, &tm_k, &k_full[st], c * 64, y, zkv);
        ++k_issued;
        if (u > 0 && !mbar_wait(&v_empty[st], (u - 1) & 1, abort, a.err)) break;
        mbar_expect_tx(&v_full[st], Cfg::kTile);
#pragma unroll
        for (int c = 0; c < kChunks; ++c)
          tma_load_3d(sV + st * Cfg::kTile + c * Cfg::kChunk, &tm_v, &v_full[st], c * 64, y, zkv);
        ++v_issued;
      }
      if (*abort) {
        // drain: copies already issued must land before the CTA exits
        for (int t = max(0, k_issued - 2); t < k_issued; ++t) {
          const unsigned long long t0 = global_ns();
          while (!mbar_try_wait(&k_full[t & 1], (t >> 1) & 1) && global_ns() - t0 < kWaitTimeoutNs) {}
        }
        for (int t = max(0, v_issued - 2); t < v_issued; ++t) {
          const unsigned long long t0 = global_ns();
          while (!mbar_try_wait(&v_full[t & 1], (t >> 1) & 1) && global_ns() - t0 < kWaitTimeoutNs) {}
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------- MMA issuer ---
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, kBN, false, false);
      constexpr uint32_t idPV = idesc_bf16_f32(128, D, false, true);
      const uint32_t q0 = smem_u32(sQ);
      bool ok = mbar_wait(q_full, 0, abort, a.err);
      auto issue_pv = [&](int u) -> bool {
        const int st = u & 1;
        if (!mbar_wait(&p_ready[st], (u >> 1) & 1, abort, a.err)) return false;
        if (!mbar_wait(&v_full[st], (u >> 1) & 1, abort, a.err)) return false;
        tc_fence_after();
        const uint32_t v0 = smem_u32(sV + st * Cfg::kTile);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint64_t bd = sw128_desc(v0 + kk * 16 * 128, Cfg::kChunk, 1024);
          mma_ts(tmem + Cfg::kO, tmem + Cfg::kP0 + st * 64 + kk * 8, bd, idPV, (u > 0 || kk > 0));
        }
        mma_commit(o_done);
        mma_commit(&v_empty[st]);
        return true;
      };
      for (int t = 0; t < nt && ok; ++t) {
        const int st = t & 1;
        if (!mbar_wait(&k_full[st], (t >> 1) & 1, abort, a.err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t k0 = smem_u32(sK + st * Cfg::kTile);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * Cfg::kChunk + (kk & 3) * 32;
          mma_ss(tmem + Cfg::kS0 + st * kBN, sw128_desc(q0 + off, 16, 1024),
                 sw128_desc(k0 + off, 16, 1024), idS, kk > 0);
        }
        mma_commit(&s_full[st]);
        mma_commit(&k_empty[st]);
        if (t > 0 && !issue_pv(t - 1)) { ok = false; break; }
      }
      if (ok && issue_pv(nt - 1)) mma_commit(o_final);
    }
  } else {
    // ------------------------------------------------------- softmax ---
    const int qw = warp & 3;             // TMEM lane quarter of this warp
    const int r = qw * 32 + lane;        // query row within the tile
    const uint32_t lane_base = static_cast<uint32_t>(qw * 32) << 16;
    const bool valid = r < nrows;
    int pos = -1, lo = 1, hi = 0;
    if (MODE == kModeGroup) {
      if (valid) {
        const size_t sidx = static_cast<size_t>(prob) * a.n + row_base + r;
        pos = a.perm[sidx];
        lo = 0;
        hi = a.farlen_slot[sidx] - 1;
      }
    } else if (valid) {
      pos = row_base + r;
      lo = MODE == kModeDense ? 0 : pos - a.w + 1;
      hi = pos;
    }
    const size_t qrow = (static_cast<size_t>(b) * a.H + h) * a.n;
    // gather this row of Q into the 128 B-swizzled K-major tile
    {
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.Q) +
                                                        (qrow + (valid ? pos : 0)) * D);
#pragma unroll
      for (int u = 0; u < D / 8; ++u) {
        const uint4 v = valid ? __ldg(src + u) : make_uint4(0, 0, 0, 0);
        const int c = u >> 3, uu = u & 7;
        *reinterpret_cast<uint4*>(sQ + c * Cfg::kChunk + r * 128 + ((uu ^ (r & 7)) << 4)) = v;
      }
      fence_proxy_async_smem();
      mbar_arrive(q_full);
    }

    float m_run = -INFINITY, l = 0.f;
    const float sl2 = a.scale_log2;
    bool ok = true;
    for (int t = 0; t < nt; ++t) {
      const int st = t & 1;
      const int j0 = (MODE == kModeGroup ? 0 : ybase) + t * kBN;
      if (!warp_wait(&s_full[st], (t >> 1) & 1, abort, a.err)) { ok = false; break; }
      tc_fence_after();
      float x[kBN];
      {
        uint32_t rr[32];
#pragma unroll
        for (int c = 0; c < kBN; c += 32) {
          tmem_ld32(tmem + lane_base + Cfg::kS0 + st * kBN + c, rr);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) x[c + e] = __uint_as_float(rr[e]);
        }
      }
      const bool full = j0 >= lo && j0 + kBN - 1 <= hi;
      if (!full) {
#pragma unroll
        for (int c = 0; c < kBN; ++c)
          if (j0 + c < lo || j0 + c > hi) x[c] = -INFINITY;
      }
      float mt = -INFINITY;
#pragma unroll
      for (int c = 0; c < kBN; ++c) mt = fmaxf(mt, x[c]);
      const float m_new = fmaxf(m_run, mt * sl2);
      const bool need = m_run != -INFINITY && m_new > m_run + kRescaleThreshold;
      if (m_run == -INFINITY) m_run = m_new;      // nothing accumulated yet for this row
      if (__any_sync(0xffffffffu, need)) {
        // O must hold every earlier PV product before it is rescaled
        if (!warp_wait(o_done, (t - 1) & 1, abort, a.err)) { ok = false; break; }
        tc_fence_after();
        const float alpha = need ? ex2f(m_run - m_new) : 1.f;
        uint32_t rr[32];
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          tmem_ld32(tmem + lane_base + Cfg::kO + c, rr);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * alpha);
          tmem_st32(tmem + lane_base + Cfg::kO + c, rr);
        }
        tmem_wait_st();
        if (need) {
          l *= alpha;
          m_run = m_new;
        }
      }
      const float mu = m_run == -INFINITY ? 0.f : m_run;
      float ls = 0.f;
      uint32_t pk[kBN / 2];
#pragma unroll
      for (int c = 0; c < kBN; c += 2) {
        const float p0 = ex2f(fmaf(x[c], sl2, -mu));
        const float p1 = ex2f(fmaf(x[c + 1], sl2, -mu));
        ls += p0 + p1;
        pk[c / 2] = pack_bf16x2(p0, p1);
      }
      l += ls;
      {
        uint32_t (&lo32)[32] = *reinterpret_cast<uint32_t(*)[32]>(&pk[0]);
        uint32_t (&hi32)[32] = *reinterpret_cast<uint32_t(*)[32]>(&pk[32]);
        tmem_st32(tmem + lane_base + Cfg::kP0 + st * 64, lo32);
        tmem_st32(tmem + lane_base + Cfg::kP0 + st * 64 + 32, hi32);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_ready[st]);
    }

    // ------------------------------------------------------ epilogue ---
    // o_done may trail by two phases here, so its parity cannot tell whether
    // the last product landed; o_final has exactly one phase.
    if (ok) ok = warp_wait(o_final, 0, abort, a.err);
    tc_fence_after();
    if (ok) {
      constexpr float kLn2 = 0.6931471805599453f;
      constexpr float kLog2e = 1.4426950408889634f;
      float c1 = l > 0.f ? 1.f / l : 0.f, c2 = 0.f;
      float lse2 = m_run + log2f(l);
      bool far = false;
      const size_t orow = (qrow + (valid ? pos : 0)) * D;
      const __nv_bfloat16* Of = static_cast<const __nv_bfloat16*>(a.O_far);
      if (MODE == kModeLocal && valid) {
        far = a.farlen_tok[static_cast<size_t>(prob) * a.n + pos] > 0;
        if (far) {
          const float lf2 = a.lse_far[qrow + pos] * kLog2e;
          const float mm = fmaxf(lse2, lf2);
          const float e1 = ex2f(lse2 - mm), e2 = ex2f(lf2 - mm);
          const float den = e1 + e2;
          c1 = e1 / (l * den);
          c2 = e2 / den;
          lse2 = mm + log2f(den);
        }
      }
      const bool write = valid && (MODE != kModeGroup || l > 0.f);
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(MODE == kModeGroup ? a.O_far : a.O);
      uint32_t rr[32];
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        tmem_ld32(tmem + lane_base + Cfg::kO + c, rr);
        tmem_wait_ld();
        if (write) {
          float f[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(rr[e]) * c1;
          if (far) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const uint4 v = *reinterpret_cast<const uint4*>(Of + orow + c + u * 8);
              const __nv_bfloat162* v2 = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 g = __bfloat1622float2(v2[e]);
                f[u * 8 + 2 * e] = fmaf(g.x, c2, f[u * 8 + 2 * e]);
                f[u * 8 + 2 * e + 1] = fmaf(g.y, c2, f[u * 8 + 2 * e + 1]);
              }
            }
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 v;
            v.x = pack_bf16x2(f[u * 8 + 0], f[u * 8 + 1]);
            v.y = pack_bf16x2(f[u * 8 + 2], f[u * 8 + 3]);
            v.z = pack_bf16x2(f[u * 8 + 4], f[u * 8 + 5]);
            v.w = pack_bf16x2(f[u * 8 + 6], f[u * 8 + 7]);
            *reinterpret_cast<uint4*>(dst + orow + c + u * 8) = v;
          }
        }
      }
      if (write) {
        if (MODE == kModeGroup) a.lse_far[qrow + pos] = lse2 * kLn2;
        else if (a.lse) a.lse[qrow + pos] = lse2 * kLn2;
      }
    }
  }

  __syncwarp();          // lanes 1..31 of warps 0 and 1 wait here for lane 0
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

// K_s[b, kv, s, :] = K[b, kv, perm_a[s], :] (and V), a = assignment of kv.
__global__ void __launch_bounds__(256) permute_kv_kernel(const uint4* __restrict__ K,
                                                         const uint4* __restrict__ V,
                                                         uint4* __restrict__ Ks,
                                                         uint4* __restrict__ Vs,
                                                         const int32_t* __restrict__ perm, int H_kv,
                                                         int n, int vec_per_row, int A,
                                                         long long total) {
  for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = e / vec_per_row;
    const int u = static_cast<int>(e % vec_per_row);
    const int s = static_cast<int>(row % n);
    const long long bk = row / n;             // b * H_kv + kv
    const int kvh = static_cast<int>(bk % H_kv);
    const long long bb = bk / H_kv;
    const long long p = bb * A + (A == 1 ? 0 : kvh);
    const int src = __ldg(perm + p * n + s);
    const long long si = (bk * n + src) * vec_per_row + u;
    Ks[e] = __ldg(K + si);
    Vs[e] = __ldg(V + si);
  }
}

template <int D>
cudaError_t launch_d(const AttnArgs& a, const CUtensorMap* tm_k, const CUtensorMap* tm_v, int mode,
                     int max_items, cudaStream_t st) {
  using Cfg = AttnCfg<D>;
  if (mode == kModeGroup) {
    const int hpa = a.A == 1 ? a.H : a.H / a.H_kv;
    const long long grid = static_cast<long long>(max_items) * hpa;
    if (grid == 0) return cudaSuccess;
    attn_tc_kernel<D, kModeGroup><<<static_cast<unsigned>(grid), 192, Cfg::kSmem, st>>>(*tm_k, *tm_v, a);
  } else {
    const long long grid = static_cast<long long>(a.B) * a.H * ((a.n + kTileM - 1) / kTileM);
    if (mode == kModeLocal)
      attn_tc_kernel<D, kModeLocal><<<static_cast<unsigned>(grid), 192, Cfg::kSmem, st>>>(*tm_k, *tm_v, a);
    else
      attn_tc_kernel<D, kModeDense><<<static_cast<unsigned>(grid), 192, Cfg::kSmem, st>>>(*tm_k, *tm_v, a);
  }
  return cudaGetLastError();
}

template <int D>
cudaError_t set_smem() {
  using Cfg = AttnCfg<D>;
  cudaError_t e;
  e = cudaFuncSetAttribute(attn_tc_kernel<D, kModeGroup>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(attn_tc_kernel<D, kModeLocal>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(attn_tc_kernel<D, kModeDense>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
}

}  // namespace

cudaError_t launch_permute_kv_bf16(const void* K, const void* V, void* Ks, void* Vs,
                                   const int32_t* perm, int B, int H_kv, int n, int d, int A,
                                   cudaStream_t st) {
  const int vpr = d / 8;
  const long long total = static_cast<long long>(B) * H_kv * n * vpr;
  if (total == 0) return cudaSuccess;
  const long long want = (total + 255) / 256;
  const int grid = static_cast<int>(want < 152LL * 16 ? want : 152LL * 16);
  permute_kv_kernel<<<grid, 256, 0, st>>>(static_cast<const uint4*>(K), static_cast<const uint4*>(V),
                                          static_cast<uint4*>(Ks), static_cast<uint4*>(Vs), perm,
                                          H_kv, n, vpr, A, total);
  return cudaGetLastError();
}

cudaError_t launch_attn_tc_bf16(const AttnArgs& a, const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                int d, int mode, int max_items, cudaStream_t st) {
  if (d == 64) return launch_d<64>(a, tm_k, tm_v, mode, max_items, st);
  if (d == 128) return launch_d<128>(a, tm_k, tm_v, mode, max_items, st);
  return cudaErrorInvalidValue;
}

cudaError_t setup_attn_kernels() {
  cudaError_t e = set_smem<64>();
  if (e != cudaSuccess) return e;
  return set_smem<128>();
}

}  // namespace focus
