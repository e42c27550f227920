// focus_assign kernels: nearest-centroid group ids.
//
// "Focus: Learning Which Attention Pairs Matter", section 2.1: each hidden
// state h_i is projected and compared with K learnable centroids; section 2.2
// and "Why Attend to Everything? Focus is the Key", section 2.3: at inference
// the assignment is hard: each token goes to its top-k centroids (k = 1 or 2).
// Per token and assignment a:
//   p = W_a h (fp32 accumulate, kept in fp32), s_k = p . c_k (fp32),
//   g = the k largest s_k, best first, the lower k first among equal scores.
//
// bf16: the projection is a [128 tokens x A*d_g] tile of h W^T on the
// tcgen05 tensor cores (TMA-fed pipeline, fp32 accumulator in TMEM); the
// epilogue reads each token's row of p from TMEM and scores the centroids
// with fp32 FMAs, or (d_g = 64, K <= 64, persistent kernel) on the tensor
// cores from p split exactly into three bf16 parts, so p is never rounded
// below fp32.  For 32, 64, 128 or 256
// projection columns the kernel is persistent: one CTA per SM streams its
// token tiles of h through a 4-6 stage TMA ring into double-buffered TMEM
// accumulators while four epilogue warps score the previous tile; wider
// projections that are a multiple of 256 columns run through the same kernel
// as passes of 256 (whole assignments each), and other widths up to 512 use
// one CTA per 128-token tile.
// fp32: one warp per token and assignment on the CUDA cores.
// With kScores the kernels write every score s_k (fp32, [B, A, n, K]) instead
// of the top-k ids: the input of the Sinkhorn soft assignment.
#include "common.cuh"
#include "kernels.h"

namespace focus {
namespace {

// Running best and runner-up over centroids scanned in increasing k: a later
// centroid displaces one only with a strictly larger score, so the lower index
// wins ties (and a NaN score never displaces anything but the empty start).
// Written as selects: the lanes of a warp disagree on which case applies.
struct Top2 {
  int b1 = -1, b2 = -1;
  float s1 = -INFINITY, s2 = -INFINITY;
  __device__ __forceinline__ void push(int k, float s) {
    const bool g1 = (b1 < 0) | (s > s1);
    const bool g2 = !g1 & ((b2 < 0) | (s > s2));
    s2 = g1 ? s1 : (g2 ? s : s2);
    b2 = g1 ? b1 : (g2 ? k : b2);
    s1 = g1 ? s : s1;
    b1 = g1 ? k : b1;
  }
};

// ------------------------------------------------------------------ fp32 ---
// One warp per (token, assignment).  Lane l accumulates projection rows
// r = l, l + 32, ... over the hidden dimension in order c = 0, 1, ... (h read
// as warp-wide broadcasts, each W row by its own lane).  Centroids then go 32
// at a time, one per lane: s_k sums p_r * c_kr in order r = 0, 1, ..., with
// p_r broadcast from its lane, and every lane replays the chunk's scores in k
// order through the same top-k update.  p and s are the sums a scalar loop
// over c and r gives, so the results do not depend on the thread layout.
constexpr int kF32Warps = 8;

template <int DG, bool kScores>
__global__ void __launch_bounds__(32 * kF32Warps) assign_f32_kernel(const float* __restrict__ h,
                                                                   const float* __restrict__ W,
                                                                   const float* __restrict__ C,
                                                                   int32_t* __restrict__ gid,
                                                                   float* __restrict__ scores, int B, int n,
                                                                   int D, int K, int A, int topk) {
  constexpr int kR = (DG + 31) / 32;   // projection rows per lane
  const int lane = lane_id();
  const int tok = blockIdx.x * kF32Warps + warp_id();
  const int a = blockIdx.y;
  if (tok >= B * n) return;            // the whole warp leaves together
  const int b = tok / n, i = tok % n;
  const float* hr = h + static_cast<size_t>(tok) * D;
  const float* Wa = W + static_cast<size_t>(a) * DG * D;
  float p[kR];
#pragma unroll
  for (int q = 0; q < kR; ++q) p[q] = 0.f;
  const bool vec = (D & 3) == 0 && (reinterpret_cast<uintptr_t>(h) & 15) == 0 &&
                   (reinterpret_cast<uintptr_t>(W) & 15) == 0;
  int c = 0;
  if (vec) {
    for (; c < D; c += 4) {
      const float4 x = __ldg(reinterpret_cast<const float4*>(hr + c));
#pragma unroll
      for (int q = 0; q < kR; ++q) {
        const int r = lane + 32 * q;
        if (r < DG) {
          const float4 wv = __ldg(reinterpret_cast<const float4*>(Wa + static_cast<size_t>(r) * D + c));
          p[q] = fmaf(wv.x, x.x, p[q]);
          p[q] = fmaf(wv.y, x.y, p[q]);
          p[q] = fmaf(wv.z, x.z, p[q]);
          p[q] = fmaf(wv.w, x.w, p[q]);
        }
      }
    }
  }
  for (; c < D; ++c) {
    const float x = __ldg(hr + c);
#pragma unroll
    for (int q = 0; q < kR; ++q) {
      const int r = lane + 32 * q;
      if (r < DG) p[q] = fmaf(__ldg(Wa + static_cast<size_t>(r) * D + c), x, p[q]);
    }
  }
  const float* Ca = C + static_cast<size_t>(a) * K * DG;
  float* srow = kScores ? scores + ((static_cast<size_t>(b) * A + a) * n + i) * K : nullptr;
  Top2 t;
  for (int k0 = 0; k0 < K; k0 += 32) {
    const int k = k0 + lane;
    const float* ck = Ca + static_cast<size_t>(k < K ? k : 0) * DG;
    float sc = 0.f;
#pragma unroll
    for (int r = 0; r < DG; ++r) sc = fmaf(__shfl_sync(0xffffffffu, p[r / 32], r % 32), __ldg(ck + r), sc);
    if (kScores) {
      if (k < K) srow[k] = sc;
    } else {
      const int nk = min(32, K - k0);
      for (int j = 0; j < nk; ++j) t.push(k0 + j, __shfl_sync(0xffffffffu, sc, j));
    }
  }
  if (!kScores && lane == 0) {
    int32_t* out = gid + ((static_cast<size_t>(b) * A + a) * n + i) * topk;
    out[0] = t.b1;
    if (topk == 2) out[1] = t.b2;
  }
}

// ------------------------------------------------------------ bf16 tcgen05 ---
constexpr int kBM = 128;          // tokens per CTA
constexpr int kBK = 64;           // hidden elements per stage (one 128 B swizzle row)

template <int NALLOC>
struct AssignCfg {
  static constexpr int kStageA = kBM * kBK * 2;            // 16 KB
  static constexpr int kStageB = NALLOC * kBK * 2;         // <= 64 KB
  static constexpr int kStage = kStageA + kStageB;
  // narrow projections: four stages and two CTAs per SM, so a whole layer's
  // tiles run in one wave and both CTAs' loads are in flight together
  static constexpr int kStages = NALLOC <= 128 ? 4 : ((196 * 1024 / kStage) > 6 ? 6 : (196 * 1024 / kStage));
  static constexpr int kSmem = kStages * kStage + 1024 /*align*/ + 256 /*barriers*/;
  static constexpr int kMinBlocks = kSmem <= 112 * 1024 ? 2 : 1;
};

template <int NALLOC, bool kScores>
__global__ void __launch_bounds__(128, AssignCfg<NALLOC>::kMinBlocks) assign_tc_kernel(
    const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_w,
    const __nv_bfloat16* __restrict__ C, int32_t* __restrict__ gid, float* __restrict__ scores,
    int B, int n, int D, int d_g, int K, int A, int topk, int* err) {
  using Cfg = AssignCfg<NALLOC>;
  constexpr int S = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * Cfg::kStage);
  uint64_t* empty = full + S;
  uint64_t* done = empty + S;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = warp_id(), lane = lane_id();
  const int ncol = A * d_g;
  const int m0 = blockIdx.x * kBM;
  const int nk = (D + kBK - 1) / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    *abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_h);
    prefetch_tmap(&tm_w);
  }
  if (warp == 1) tmem_alloc(tmem_slot, NALLOC);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // producer: h tile [128 x 64] and W tile [ncol x 64] per stage; W rows come
    // in boxes of wbox rows (the tensor map's box height)
    const int wbox = ncol < 256 ? ncol : 256;
    const int wloads = (ncol + wbox - 1) / wbox;
    const uint32_t bytes = Cfg::kStageA + wloads * wbox * kBK * 2;
    int issued = 0;
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % S, u = kb / S;
      if (u > 0 && !mbar_wait(&empty[s], (u - 1) & 1, abort, err)) break;
      uint8_t* sa = smem + s * Cfg::kStage;
      uint8_t* sb = sa + Cfg::kStageA;
      mbar_expect_tx(&full[s], bytes);
      tma_load_2d(sa, &tm_h, &full[s], kb * kBK, m0);
      for (int l = 0; l < wloads; ++l) tma_load_2d(sb + l * wbox * 128, &tm_w, &full[s], kb * kBK, l * wbox);
      ++issued;
    }
    if (*abort) {
      // let copies already in flight land before the CTA exits
      for (int kb = max(0, issued - S); kb < issued; ++kb) {
        if (!mbar_wait(&full[kb % S], (kb / S) & 1, abort, err)) {
          // the abort flag is already up; a bounded wait on the timer remains
          const unsigned long long t0 = global_ns();
          while (!mbar_try_wait(&full[kb % S], (kb / S) & 1) && global_ns() - t0 < kWaitTimeoutNs) {}
        }
      }
    }
  } else if (warp == 1 && lane == 0) {
    // MMA issuer: D[128 x ncol] += h_tile * W_tile^T, N split in <= 256 chunks
    bool ok = true;
    for (int kb = 0; kb < nk && ok; ++kb) {
      const int s = kb % S, u = kb / S;
      if (!mbar_wait(&full[s], u & 1, abort, err)) { ok = false; break; }
      tc_fence_after();
      const uint32_t sa = smem_u32(smem + s * Cfg::kStage);
      const uint32_t sb = sa + Cfg::kStageA;
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk) {
        const uint64_t ad = sw128_desc(sa + kk * 32, 16, 1024);
        for (int c0 = 0; c0 < ncol; c0 += 256) {
          const int nn = min(256, ncol - c0);
          const uint64_t bd = sw128_desc(sb + c0 * 128 + kk * 32, 16, 1024);
          mma_ss(tmem + c0, ad, bd, idesc_bf16_f32(128, nn, false, false), (kb | kk) != 0);
        }
      }
      mma_commit(&empty[s]);
    }
    mma_commit(done);
  }
  __syncwarp();

  // epilogue (all 4 warps): warp w owns TMEM lanes 32w..32w+31 = tokens m0+32w+lane
  const bool got = mbar_wait(done, 0, abort, err);
  tc_fence_after();
  __syncthreads();   // pipeline smem is free from here on: reuse it for centroids
  float* Cs = reinterpret_cast<float*>(smem);
  const int kc = (S * Cfg::kStage) / (d_g * 4);   // centroids per shared-memory chunk
  const int row = warp * 32 + lane;
  const int tok = m0 + row;
  for (int a = 0; a < A; ++a) {
    float p[128];
#pragma unroll
    for (int c = 0; c < 128; c += 32) {
      if (c < d_g) {
        uint32_t r[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + a * d_g + c, r);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) p[c + j] = __uint_as_float(r[j]);
      }
    }
    Top2 t;
    const bool keep = got && !*abort && tok < B * n;
    float* srow = kScores && keep
                      ? scores + ((static_cast<size_t>(tok / n) * A + a) * n + tok % n) * K
                      : nullptr;
    for (int k0 = 0; k0 < K; k0 += kc) {
      const int kn = min(kc, K - k0);
      __syncthreads();
      for (int e = threadIdx.x; e < kn * d_g; e += blockDim.x)
        Cs[e] = __bfloat162float(C[(static_cast<size_t>(a) * K + k0) * d_g + e]);
      __syncthreads();
      int k = 0;
      // four centroids per pass: independent FMA chains, 16-byte broadcast reads;
      // each score still sums j = 0, 1, ... in order
      for (; k + 4 <= kn; k += 4) {
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 128; j += 4) {
          if (j < d_g) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float4 c4 = *reinterpret_cast<const float4*>(Cs + (k + q) * d_g + j);
              sc[q] = fmaf(p[j], c4.x, sc[q]);
              sc[q] = fmaf(p[j + 1], c4.y, sc[q]);
              sc[q] = fmaf(p[j + 2], c4.z, sc[q]);
              sc[q] = fmaf(p[j + 3], c4.w, sc[q]);
            }
          }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (kScores) {
            if (srow) srow[k0 + k + q] = sc[q];
          } else {
            t.push(k0 + k + q, sc[q]);
          }
        }
      }
      for (; k < kn; ++k) {
        const float* ck = Cs + k * d_g;
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < 128; ++j)
          if (j < d_g) s = fmaf(p[j], ck[j], s);
        if (kScores) {
          if (srow) srow[k0 + k] = s;
        } else {
          t.push(k0 + k, s);
        }
      }
    }
    if (!kScores && keep) {
      const int b = tok / n, i = tok % n;
      int32_t* out = gid + ((static_cast<size_t>(b) * A + a) * n + i) * topk;
      out[0] = t.b1;
      if (topk == 2) out[1] = t.b2;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, NALLOC);
  }
}

// ------------------------------------------------ bf16 tcgen05, persistent ---
// One CTA per SM walks tiles blockIdx.x, blockIdx.x + gridDim.x, ...  Warp 0
// issues the TMA loads of every (tile, k-step) into a kStages ring, warp 1 the
// MMAs into TMEM buffer (tile index & 1), and warps 2-5 (one per TMEM lane
// quadrant) score a tile once its accumulator is complete, releasing the
// buffer as soon as they have read it.  The centroids are staged in shared
// memory as fp32, one chunk [d_g][chunk] at a time (kept while it stays the
// same), and every lane reads the same address (broadcast) while scoring two
// centroids per packed FMA.
constexpr int kStreamThreads = 192;

template <int NALLOC>
struct StreamCfg {
  // 64-column k-slabs per stage: two for narrow projections, so each stage
  // asks for 256 contiguous bytes of every h row at once
  static constexpr int kSlabs = NALLOC <= 64 ? 2 : 1;
  static constexpr int kSlabA = kBM * kBK * 2;             // 16 KB of h per slab
  static constexpr int kSlabB = NALLOC * kBK * 2;          // <= 32 KB of W per slab
  static constexpr int kStageA = kSlabs * kSlabA;
  static constexpr int kStageB = kSlabs * kSlabB;
  static constexpr int kStage = kStageA + kStageB;
  static constexpr int kStages = (200 * 1024 / kStage) < 8 ? (200 * 1024 / kStage) : 8;
  static constexpr int kRing = kStages * kStage;
  // fp32 centroids for the scoring loop, in what the 227 KB opt-in leaves
  // (24-32 KB): a chunk of centroids [d_g][chunk] per fill
  static constexpr int kCLeft = 227 * 1024 - kRing - 1024 /*align*/ - 256 /*barriers*/;
  static constexpr int kCBytes = (kCLeft > 32768 ? 32768 : kCLeft) & ~1023;
  static constexpr int kSmem = kRing + 1024 + 256 + kCBytes;
  static constexpr int kTmemCols = 2 * NALLOC;              // two accumulators
};

// Scores of 32 centroids kb .. kb + 31 of a staged chunk (cs[j * kc + k],
// fp32): acc holds them as pairs (k, k + 1); each score is summed from 0 in
// order j = 0, 1, ... with one rounding per FMA, as a scalar loop would.
template <int DG>
__device__ __forceinline__ void score32(const float (&p)[128], const float* cs, int kc, int kb,
                                        uint64_t (&acc)[16]) {
#pragma unroll
  for (int q = 0; q < 16; ++q) acc[q] = 0ull;
#pragma unroll
  for (int j = 0; j < DG; ++j) {
    const uint64_t pp = f2_pack(p[j], p[j]);
    const float* row = cs + j * kc + kb;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      uint64_t c0, c1;
      lds_f2x2(row + 4 * q, c0, c1);
      acc[2 * q] = f2_fma(pp, c0, acc[2 * q]);
      acc[2 * q + 1] = f2_fma(pp, c1, acc[2 * q + 1]);
    }
  }
}

template <int NALLOC, int DG, bool kScores>
__global__ void __launch_bounds__(kStreamThreads, 1) assign_stream_kernel(
    const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_w,
    const __nv_bfloat16* __restrict__ C, int32_t* __restrict__ gid, float* __restrict__ scores,
    int B, int n, int D, int K, int A, int topk, int R, int a0, int npass, int A_all, int* err) {
  // this launch covers assignments a0 .. a0 + npass * A - 1 of A_all in npass
  // passes of A: unit u is token tile u / npass in pass u % npass (W rows from
  // (a0 + pass * A) * DG), so the passes over one tile run side by side on
  // neighbouring CTAs and all but the first read its h rows from L2
  using Cfg = StreamCfg<NALLOC>;
  constexpr int S = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * Cfg::kStage);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;      // [2] accumulator complete
  uint64_t* tfree = tfull + 2;      // [2] accumulator read out (4 epilogue warps)
  uint64_t* sc_bar = tfree + 2;     // scoring product done (tensor-core scores)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sc_bar + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = warp_id(), lane = lane_id();
  const int ncol = A * DG;
  const int ntiles = (B * n + R - 1) / R;   // tiles of R <= 128 tokens
  const int nunits = ntiles * npass;
  const int nk = (D + kBK - 1) / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tfree[b], 4);
    }
    mbar_init(sc_bar, 1);
    *abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_h);
    prefetch_tmap(&tm_w);
  }
  if (warp == 1) tmem_alloc(tmem_slot, Cfg::kTmemCols);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // a tile's R rows of h fill the first R rows of each slab; the MMAs read
      // all 128, and the accumulator rows past R are never read out
      const uint32_t slab_bytes = R * kBK * 2 + ncol * kBK * 2;
      const int ns = (nk + Cfg::kSlabs - 1) / Cfg::kSlabs;   // stages per tile
      int it = 0;
      bool ok = true;
      for (int unit = blockIdx.x; unit < nunits && ok; unit += gridDim.x) {
        const int tile = unit / npass, wrow = (a0 + (unit % npass) * A) * DG;
        for (int ks = 0; ks < ns; ++ks, ++it) {
          const int s = it % S, u = it / S;
          if (u > 0 && !mbar_wait_nap(&empty[s], (u - 1) & 1, abort, err)) { ok = false; break; }
          uint8_t* sa = smem + s * Cfg::kStage;
          const int nsl = min(Cfg::kSlabs, nk - ks * Cfg::kSlabs);
          mbar_expect_tx(&full[s], slab_bytes * nsl);
          for (int j = 0; j < nsl; ++j) {
            const int kb = ks * Cfg::kSlabs + j;
            tma_load_2d(sa + j * Cfg::kSlabA, &tm_h, &full[s], kb * kBK, tile * R);
            tma_load_2d(sa + Cfg::kStageA + j * Cfg::kSlabB, &tm_w, &full[s], kb * kBK, wrow);
          }
        }
      }
      if (*abort || !ok) {
        // let copies already in flight land before the CTA exits
        for (int j = max(0, it - S); j < it; ++j) {
          const unsigned long long t0 = global_ns();
          while (!mbar_try_wait(&full[j % S], (j / S) & 1) && global_ns() - t0 < kWaitTimeoutNs) {}
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idn = idesc_bf16_f32(128, NALLOC, false, false);
      int it = 0;
      bool ok = true;
      for (int unit = blockIdx.x, i = 0; unit < nunits && ok; unit += gridDim.x, ++i) {
        const int buf = i & 1;
        if (i >= 2 && !mbar_wait_nap(&tfree[buf], ((i >> 1) - 1) & 1, abort, err)) break;
        const int ns = (nk + Cfg::kSlabs - 1) / Cfg::kSlabs;
        for (int ks = 0; ks < ns; ++ks, ++it) {
          const int s = it % S, u = it / S;
          if (!mbar_wait_nap(&full[s], u & 1, abort, err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * Cfg::kStage);
          const int nsl = min(Cfg::kSlabs, nk - ks * Cfg::kSlabs);
          for (int j = 0; j < nsl; ++j) {
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              mma_ss(tmem + buf * NALLOC, sw128_desc(sa + j * Cfg::kSlabA + kk * 32, 16, 1024),
                     sw128_desc(sa + Cfg::kStageA + j * Cfg::kSlabB + kk * 32, 16, 1024), idn,
                     (ks | j | kk) != 0);
          }
          mma_commit(&empty[s]);
        }
        if (ok) mma_commit(&tfull[buf]);
      }
    }
  } else {
    // epilogue: warps 2-5 read TMEM lane quadrants 2, 3, 0, 1
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int et = threadIdx.x - 64;   // 0..127 over the epilogue warps
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    // centroids in chunks of kc (a multiple of 32) staged as fp32 [DG][kc];
    // a chunk stays staged while consecutive tiles use the same one
    float* cs = reinterpret_cast<float*>(smem + Cfg::kRing + 256);
    const int kc_max = (Cfg::kCBytes / 4 / DG) & ~31;
    const int kc = min(kc_max, (K + 31) & ~31);
    int staged_a = -1, staged_k0 = -1;
    // d_g = 64 and K <= 64: the scores on the tensor cores instead.  p (fp32)
    // splits exactly into three bf16 parts, p = hi + mid + lo (each part is
    // the rounding of what the parts before it leave, and what is left after
    // two parts has at most 8 significant bits); the three parts go through one
    // 16 KB operand slab in turn, each multiplied with the centroids (bf16,
    // exact in the product) into the assignment's own 64 accumulator columns,
    // which p has been read out of.  Products are exact and accumulate in
    // fp32, so the scores are fp32 dot products of the fp32 p with the
    // centroids, summed in the tensor core's order.
    const bool tc = DG == 64 && K <= 64;
    uint8_t* As = smem + Cfg::kRing + 1024;   // 128 rows x 128 B, 128-byte swizzle
    uint8_t* Bs = As + 128 * 128;             // N rows x 128 B: the centroids
    uint32_t sc_ph = 0;
    bool fine = true;
    for (int unit = blockIdx.x, i = 0; unit < nunits && fine; unit += gridDim.x, ++i) {
      const int buf = i & 1;
      // every epilogue thread leaves the loop together, so the named barriers
      // below always see all 128
      if (!named_barrier_and(1, 128, mbar_wait(&tfull[buf], (i >> 1) & 1, abort, err))) break;
      tc_fence_after();
      const int tile = unit / npass, pa = a0 + (unit % npass) * A;   // the pass's first assignment
      const int tok = tile * R + row;
      const bool keep = row < R && tok < B * n;
      const int b = keep ? tok / n : 0, ti = keep ? tok % n : 0;
      for (int a = 0; a < A; ++a) {
        float p[128];
#pragma unroll
        for (int c = 0; c < DG; c += 32) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_base + buf * NALLOC + a * DG + c, r);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) p[c + j] = __uint_as_float(r[j]);
        }
        if (!tc && a == A - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tfree[buf]);   // the accumulator may take tile i + 2
        }
        const __nv_bfloat16* Ca = C + static_cast<size_t>(pa + a) * K * DG;
        float* srow = kScores && keep ? scores + ((static_cast<size_t>(b) * A_all + pa + a) * n + ti) * K : nullptr;
        Top2 t;
        if constexpr (DG == 64) {
          if (tc) {
            const int N = (K + 15) & ~15;
            const bool stage_b = staged_a != pa + a;
            uint4 cw[4];
            if (stage_b) {
#pragma unroll
              for (int f = 0; f < 4; ++f) {
                const int e = et + 128 * f, k = e >> 3, ch = e & 7;
                cw[f] = make_uint4(0u, 0u, 0u, 0u);
                if (k < K) cw[f] = __ldg(reinterpret_cast<const uint4*>(Ca + static_cast<size_t>(k) * 64 + ch * 8));
              }
            }
            for (int part = 0; part < 3 && fine; ++part) {
              uint32_t w[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const uint32_t v = pack_bf16x2(p[2 * j], p[2 * j + 1]);
                w[j] = v;
                p[2 * j] -= __uint_as_float(v << 16);
                p[2 * j + 1] -= __uint_as_float(v & 0xffff0000u);
              }
              if (part == 0 && stage_b) {
#pragma unroll
                for (int f = 0; f < 4; ++f) {
                  const int e = et + 128 * f, k = e >> 3, ch = e & 7;
                  if (k < N) *reinterpret_cast<uint4*>(Bs + k * 128 + ((ch ^ (k & 7)) << 4)) = cw[f];
                }
              }
#pragma unroll
              for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4*>(As + row * 128 + ((c ^ (row & 7)) << 4)) =
                    make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
              fence_proxy_async_smem();
              tc_fence_before();
              named_barrier(1, 128);
              if (et == 0) {
                tc_fence_after();
                const uint32_t idn = idesc_bf16_f32(128, N, false, false);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  mma_ss(tmem + buf * NALLOC + a * 64, sw128_desc(smem_u32(As) + kk * 32, 16, 1024),
                         sw128_desc(smem_u32(Bs) + kk * 32, 16, 1024), idn, (part | kk) != 0);
                mma_commit(sc_bar);
              }
              // a short wait: poll with naps (a suspend hint can sleep past the commit)
              fine = named_barrier_and(1, 128, mbar_wait_nap(sc_bar, sc_ph & 1, abort, err));
              ++sc_ph;
              tc_fence_after();
            }
            if (!fine) break;
            staged_a = pa + a;
            // the scores: columns k < K of the assignment's accumulator block
#pragma unroll
            for (int c = 0; c < 64; c += 32) {
              if (c < N) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_base + buf * NALLOC + a * 64 + c, r);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                  const int k = c + j;
                  if (k < K) {
                    if (kScores) {
                      if (srow) srow[k] = __uint_as_float(r[j]);
                    } else {
                      t.push(k, __uint_as_float(r[j]));
                    }
                  }
                }
              }
            }
            if (a == A - 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&tfree[buf]);   // the accumulator may take tile i + 2
            }
            if (!kScores && keep) {
              int32_t* out = gid + ((static_cast<size_t>(b) * A_all + pa + a) * n + ti) * topk;
              out[0] = t.b1;
              if (topk == 2) out[1] = t.b2;
            }
            continue;
          }
        }
        for (int k0 = 0; k0 < K; k0 += kc) {
          const int nk = min(kc, K - k0);
          if (staged_a != pa + a || staged_k0 != k0) {
            named_barrier(1, 128);   // the previous chunk is no longer read
            // eight 16-byte loads per thread in flight, then their stores
            constexpr int kFill = 8;
            for (int e0 = et; e0 < kc * (DG / 8); e0 += 128 * kFill) {
              uint4 w[kFill];
#pragma unroll
              for (int f = 0; f < kFill; ++f) {
                const int e = e0 + f * 128, kk = e / (DG / 8), j8 = (e % (DG / 8)) * 8;
                w[f] = make_uint4(0u, 0u, 0u, 0u);
                if (e < kc * (DG / 8) && kk < nk)
                  w[f] = __ldg(reinterpret_cast<const uint4*>(Ca + static_cast<size_t>(k0 + kk) * DG + j8));
              }
#pragma unroll
              for (int f = 0; f < kFill; ++f) {
                const int e = e0 + f * 128, kk = e / (DG / 8), j8 = (e % (DG / 8)) * 8;
                if (e >= kc * (DG / 8)) break;
                const uint32_t u[4] = {w[f].x, w[f].y, w[f].z, w[f].w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  cs[(j8 + 2 * q) * kc + kk] = __uint_as_float(u[q] << 16);
                  cs[(j8 + 2 * q + 1) * kc + kk] = __uint_as_float(u[q] & 0xffff0000u);
                }
              }
            }
            named_barrier(1, 128);
            staged_a = pa + a;
            staged_k0 = k0;
          }
          for (int kb = 0; kb < nk; kb += 32) {
            uint64_t acc[16];
            score32<DG>(p, cs, kc, kb, acc);
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              float s0, s1;
              f2_unpack(acc[q], s0, s1);
              const int k = k0 + kb + 2 * q;
              if (kb + 2 * q < nk) {
                if (kScores) {
                  if (srow) srow[k] = s0;
                } else {
                  t.push(k, s0);
                }
              }
              if (kb + 2 * q + 1 < nk) {
                if (kScores) {
                  if (srow) srow[k + 1] = s1;
                } else {
                  t.push(k + 1, s1);
                }
              }
            }
          }
        }
        if (!kScores && keep) {
          int32_t* out = gid + ((static_cast<size_t>(b) * A_all + pa + a) * n + ti) * topk;
          out[0] = t.b1;
          if (topk == 2) out[1] = t.b2;
        }
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

template <int NALLOC, int DG>
cudaError_t launch_stream(const AssignLaunch& L, const CUtensorMap* tm_h, const CUtensorMap* tm_w,
                          int a0, int A_pass, int npass, cudaStream_t st) {
  using Cfg = StreamCfg<NALLOC>;
  const int R = L.tile_rows;
  if (R < 1 || R > kBM || npass < 1) return cudaErrorInvalidValue;
  const long long units = static_cast<long long>((L.B * L.n + R - 1) / R) * npass;
  const int grid = static_cast<int>(units < L.num_sms ? units : L.num_sms);
  const __nv_bfloat16* C = static_cast<const __nv_bfloat16*>(L.C);
  if (L.scores)
    assign_stream_kernel<NALLOC, DG, true><<<grid, kStreamThreads, Cfg::kSmem, st>>>(
        *tm_h, *tm_w, C, L.gid, L.scores, L.B, L.n, L.D, L.K, A_pass, L.topk, R, a0, npass, L.A, L.err);
  else
    assign_stream_kernel<NALLOC, DG, false><<<grid, kStreamThreads, Cfg::kSmem, st>>>(
        *tm_h, *tm_w, C, L.gid, L.scores, L.B, L.n, L.D, L.K, A_pass, L.topk, R, a0, npass, L.A, L.err);
  return cudaGetLastError();
}

template <int NALLOC>
cudaError_t launch_stream_dg(const AssignLaunch& L, const CUtensorMap* tm_h, const CUtensorMap* tm_w,
                             int a0, int A_pass, int npass, cudaStream_t st) {
  // an assignment's d_g columns fit the accumulator (NALLOC >= d_g)
  if constexpr (NALLOC >= 32)
    if (L.d_g == 32) return launch_stream<NALLOC, 32>(L, tm_h, tm_w, a0, A_pass, npass, st);
  if constexpr (NALLOC >= 64)
    if (L.d_g == 64) return launch_stream<NALLOC, 64>(L, tm_h, tm_w, a0, A_pass, npass, st);
  if constexpr (NALLOC >= 128)
    if (L.d_g == 128) return launch_stream<NALLOC, 128>(L, tm_h, tm_w, a0, A_pass, npass, st);
  return cudaErrorInvalidValue;
}

template <int NALLOC>
cudaError_t launch_tc(const AssignLaunch& L, const CUtensorMap* tm_h, const CUtensorMap* tm_w,
                      cudaStream_t st) {
  if (L.tile_rows != kBM) return cudaErrorInvalidValue;
  const int grid = (L.B * L.n + kBM - 1) / kBM;
  if (L.scores)
    assign_tc_kernel<NALLOC, true><<<grid, 128, AssignCfg<NALLOC>::kSmem, st>>>(
        *tm_h, *tm_w, static_cast<const __nv_bfloat16*>(L.C), L.gid, L.scores, L.B, L.n, L.D,
        L.d_g, L.K, L.A, L.topk, L.err);
  else
    assign_tc_kernel<NALLOC, false><<<grid, 128, AssignCfg<NALLOC>::kSmem, st>>>(
        *tm_h, *tm_w, static_cast<const __nv_bfloat16*>(L.C), L.gid, L.scores, L.B, L.n, L.D,
        L.d_g, L.K, L.A, L.topk, L.err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_assign_f32(const AssignLaunch& L, cudaStream_t st) {
  const dim3 grid((L.B * L.n + kF32Warps - 1) / kF32Warps, L.A);
  constexpr int kThreadsF32 = 32 * kF32Warps;
  const float* h = static_cast<const float*>(L.h);
  const float* W = static_cast<const float*>(L.W);
  const float* C = static_cast<const float*>(L.C);
  switch (L.d_g) {
    case 16:
      if (L.scores) assign_f32_kernel<16, true><<<grid, kThreadsF32, 0, st>>>(h, W, C, L.gid, L.scores, L.B, L.n, L.D, L.K, L.A, L.topk);
      else assign_f32_kernel<16, false><<<grid, kThreadsF32, 0, st>>>(h, W, C, L.gid, L.scores, L.B, L.n, L.D, L.K, L.A, L.topk);
      break;
    case 32:
      if (L.scores) assign_f32_kernel<32, true><<<grid, kThreadsF32, 0, st>>>(h, W, C, L.gid, L.scores, L.B, L.n, L.D, L.K, L.A, L.topk);
      else assign_f32_kernel<32, false><<<grid, kThreadsF32, 0, st>>>(h, W, C, L.gid, L.scores, L.B, L.n, L.D, L.K, L.A, L.topk);
      break;
    case 64:
      if (L.scores) assign_f32_kernel<64, true><<<grid, kThreadsF32, 0, st>>>(h, W, C, L.gid, L.scores, L.B, L.n, L.D, L.K, L.A, L.topk);
      else assign_f32_kernel<64, false><<<grid, kThreadsF32, 0, st>>>(h, W, C, L.gid, L.scores, L.B, L.n, L.D, L.K, L.A, L.topk);
      break;
    case 128:
      if (L.scores) assign_f32_kernel<128, true><<<grid, kThreadsF32, 0, st>>>(h, W, C, L.gid, L.scores, L.B, L.n, L.D, L.K, L.A, L.topk);
      else assign_f32_kernel<128, false><<<grid, kThreadsF32, 0, st>>>(h, W, C, L.gid, L.scores, L.B, L.n, L.D, L.K, L.A, L.topk);
      break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

static bool stream_width(int ncol) { return ncol == 32 || ncol == 64 || ncol == 128 || ncol == 256; }
// wider projections run as passes of 256 columns (whole assignments each)
static bool stream_passes(int ncol) { return ncol > 256 && ncol % 256 == 0; }

int assign_tile_rows(int tokens, int ncol, int num_sms) {
  // With t tiles per SM the last wave is full when every tile has the same
  // share of the tokens: R = ceil(tokens / (SMs * t)), which lies in (64, 128]
  // for t >= 2.  One tile per SM or less keeps 128-token tiles.
  if (!(stream_width(ncol) || stream_passes(ncol)) || num_sms < 1) return kBM;
  const long long per_wave = static_cast<long long>(num_sms) * kBM;
  if (tokens <= per_wave) return kBM;
  const long long t = (tokens + per_wave - 1) / per_wave;
  const long long span = static_cast<long long>(num_sms) * t;
  return static_cast<int>((tokens + span - 1) / span);
}

cudaError_t launch_assign_bf16(const AssignLaunch& L, const CUtensorMap* tm_h,
                               const CUtensorMap* tm_w, cudaStream_t st) {
  // the persistent kernel loads W in one box per stage: ncol is its exact width
  const int ncol = L.A * L.d_g;
  if (ncol == 32) return launch_stream_dg<32>(L, tm_h, tm_w, 0, L.A, 1, st);
  if (ncol == 64) return launch_stream_dg<64>(L, tm_h, tm_w, 0, L.A, 1, st);
  if (ncol == 128) return launch_stream_dg<128>(L, tm_h, tm_w, 0, L.A, 1, st);
  if (ncol == 256) return launch_stream_dg<256>(L, tm_h, tm_w, 0, L.A, 1, st);
  if (stream_passes(ncol)) {
    // 256 columns (256 / d_g assignments) per pass, each pass keeping the
    // two-accumulator pipeline of the 256-wide kernel; one launch walks (tile,
    // pass) units with the passes of a tile side by side, so h streams from
    // HBM about once
    const int per = 256 / L.d_g;
    return launch_stream_dg<256>(L, tm_h, tm_w, 0, per, L.A / per, st);
  }
  if (ncol <= 32) return launch_tc<32>(L, tm_h, tm_w, st);
  if (ncol <= 64) return launch_tc<64>(L, tm_h, tm_w, st);
  if (ncol <= 128) return launch_tc<128>(L, tm_h, tm_w, st);
  if (ncol <= 256) return launch_tc<256>(L, tm_h, tm_w, st);
  if (ncol <= 512) return launch_tc<512>(L, tm_h, tm_w, st);
  return cudaErrorInvalidValue;
}

cudaError_t setup_assign_kernels() {
  cudaError_t e;
#define FOCUS_SET_SMEM(N)                                                                          \
  e = cudaFuncSetAttribute(assign_tc_kernel<N, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                           AssignCfg<N>::kSmem);                                                   \
  if (e != cudaSuccess) return e;                                                                  \
  e = cudaFuncSetAttribute(assign_tc_kernel<N, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,  \
                           AssignCfg<N>::kSmem);                                                   \
  if (e != cudaSuccess) return e;
  FOCUS_SET_SMEM(32)
  FOCUS_SET_SMEM(64)
  FOCUS_SET_SMEM(128)
  FOCUS_SET_SMEM(256)
  FOCUS_SET_SMEM(512)
#undef FOCUS_SET_SMEM
#define FOCUS_SET_SMEM2(N, G)                                                                       \
  e = cudaFuncSetAttribute(assign_stream_kernel<N, G, false>,                                       \
                           cudaFuncAttributeMaxDynamicSharedMemorySize, StreamCfg<N>::kSmem);       \
  if (e != cudaSuccess) return e;                                                                  \
  e = cudaFuncSetAttribute(assign_stream_kernel<N, G, true>,                                        \
                           cudaFuncAttributeMaxDynamicSharedMemorySize, StreamCfg<N>::kSmem);       \
  if (e != cudaSuccess) return e;
  FOCUS_SET_SMEM2(32, 32)
  FOCUS_SET_SMEM2(64, 32)
  FOCUS_SET_SMEM2(64, 64)
  FOCUS_SET_SMEM2(128, 32)
  FOCUS_SET_SMEM2(128, 64)
  FOCUS_SET_SMEM2(128, 128)
  FOCUS_SET_SMEM2(256, 32)
  FOCUS_SET_SMEM2(256, 64)
  FOCUS_SET_SMEM2(256, 128)
#undef FOCUS_SET_SMEM2
  return cudaSuccess;
}

}  // namespace focus
