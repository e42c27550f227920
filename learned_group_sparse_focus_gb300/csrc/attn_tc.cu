// Focus attention on the tcgen05 tensor cores (bf16 in, fp32 accumulate).
//
// "Focus: Learning Which Attention Pairs Matter", section 2.1: local window
// pairs at full resolution, far pairs only inside a group; section 2.2: far
// pairs of different groups are skipped outright; section 3.3 and "Why Attend
// to Everything? Focus is the Key", section 2.3: the pattern splits into a
// local-window attention and an in-group causal attention whose softmaxes
// combine exactly ("Why Attend to Everything?", section 2.1).
//
// One persistent kernel, three modes.  A work unit is 256 query rows split in
// two 128-row halves (A and B) that share every K/V tile:
//   group  a work item: <= 256 sorted slots of one group; keys are the group's
//          earlier members at or before i - w (slot < farlen of the row), read
//          from K/V pre-permuted into sorted order so each key tile is one
//          dense TMA box.  Writes the normalised partial O and its LSE at each
//          row's token position.
//   local  256 consecutive tokens, keys j in [i - w + 1, i]; merges the group
//          partial by log-sum-exp when the row has far keys; writes O.
//   dense  256 consecutive tokens, every j <= i (the comparator).
//
// Warp roles (384 threads), one CTA per SM looping over units:
//   warps 0-3   softmax of half A, one query row per thread
//   warps 4-7   softmax of half B
//   warp 8      loads: Q halves (TMA, or a cp.async row gather through perm in
//               group mode) and K/V tiles (TMA, 2-stage rings)
//   warp 9      TMEM owner and MMA issuer.  Per key tile t it issues
//               PV_A(t), S_A(t+1), PV_B(t), S_B(t+1), so each half's softmax
//               overlaps the other half's MMAs (ping-pong), and S_X(t+1)
//               lands only after PV_X(t): a softmax that sees S_X(t+1) knows
//               O_X already holds every earlier product.
//   warps 10-11 idle: they complete warpgroup 2 for the register split
// Softmax: S from TMEM, keep rule applied to boundary tiles in registers,
// online max/sum in fp32 (exp2 domain), P written back as bf16 over S's own
// TMEM columns, O rescaled in TMEM only when the running max grows by more
// than 2^8; the epilogue normalises (and merges) O straight from TMEM while the
// MMA warp already runs the next unit's first S products.
// TMEM (512 columns): S/P of half X at 128*X, O of half X at 256 + 128*X.
// Every wait is bounded; on timeout the CTA raises an error bit, drains its
// copies, frees TMEM and exits.
#include "common.cuh"
#include "kernels.h"

namespace focus {
namespace {

constexpr int kBN = 128;                     // keys per tile
constexpr int kHalf = 128;                   // query rows per half
constexpr int kUnitRows = 2 * kHalf;
constexpr float kRescaleThreshold = 8.0f;    // log2 units
constexpr int kThreads = 384;
// K and V tiles share one ring of 32 KB slots (K(t) then V(t)), five deep:
// the loader runs about 2.5 tiles ahead of the MMAs, enough to cover a TMA
// round trip while every SM streams keys at once.
constexpr int kKvSlots = 5;
// Register split (setmaxnreg).  The kernel launches at 168 registers per
// thread (384 x 168 = 64512, the cap for 12 warps).  Warpgroup 2 (loads, MMA,
// two idle warps) gives registers back down to 88 and the two softmax
// warpgroups take them up to 208: 4*32*88 + 8*32*208 = 64512, and each SM
// sub-partition then holds 208 + 208 + 88 = 504 registers per lane (<= 512).
constexpr int kRegsLow = 88;
constexpr int kRegsHigh = 208;

template <int D>
struct AttnCfg {
  static constexpr int kChunk = 128 * 128;   // 64 columns x 128 rows, one swizzle slab
  static constexpr int kTile = 128 * D * 2;  // one 128-row Q/K/V tile
  static constexpr int kQ = 0;               // two halves
  static constexpr int kRing = kQ + 2 * kTile;           // K/V slots
  static constexpr int kBar = kRing + kKvSlots * kTile;
  static constexpr int kSmem = kBar + 512 + 1024;
  static constexpr uint32_t kTmemCols = 512;
};

// Tuning knobs (compile time).  FOCUS_EXP_POLY_PER8: of every 8 columns of a
// fully kept tile, how many take exp2 on the FMA pipe (exp2_poly) instead of
// the MUFU unit, which two softmax warpgroups otherwise saturate.
#ifndef FOCUS_EXP_POLY_PER8
#define FOCUS_EXP_POLY_PER8 0
#endif

// 2^t on the FMA pipe (Cody-Waite style split): t = j + f with j = round(t)
// and |f| <= 1/2; 2^f from a cubic fitted here for relative error on
// [-1/2, 1/2] by iteratively reweighted least squares (max relative error
// 1.3e-4, well below the bf16 rounding P receives); 2^j added to the exponent
// field.  t is clamped at -126 so the result stays a normal float, so callers
// use it only on columns that are kept (a masked column must give exactly 0).
__device__ __forceinline__ float exp2_poly(float t) {
  constexpr float kRound = 12582912.f;   // 1.5 * 2^23: t + kRound holds round(t) in its low bits
  constexpr float c1 = 0.6932254433631897f, c2 = 0.24229750037193298f, c3 = 0.05533519387245178f;
  t = fmaxf(t, -126.f);
  const float r = t + kRound;
  const float f = t - (r - kRound);
  const float p = fmaf(fmaf(fmaf(c3, f, c2), f, c1), f, 1.f);
  return __int_as_float(__float_as_int(p) + (__float_as_int(r) << 23));
}

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

struct Unit {
  int b, h, prob, zkv, zq, ybase;
  int row0[2], nrows[2];
  int t0[2], t1[2];   // inclusive key-tile range of each half; t1 < t0: half idle
  int T0, T1;
};

__device__ __forceinline__ bool active(const Unit& U, int x) { return U.t1[x] >= U.t0[x]; }
__device__ __forceinline__ bool active_at(const Unit& U, int x, int t) {
  return t >= U.t0[x] && t <= U.t1[x];
}

template <int MODE>
__device__ __forceinline__ int unit_count(const AttnArgs& a) {
  if (MODE == kModeGroup) {
    const int hpa = a.A == 1 ? a.H : a.H / a.H_kv;
    return *a.n_items * hpa;
  }
  return a.B * a.H * ((a.n + kUnitRows - 1) / kUnitRows);
}

template <int MODE>
__device__ __forceinline__ void decode_unit(const AttnArgs& a, int u, Unit& U) {
  int kv, asg;
  if (MODE == kModeGroup) {
    const int hpa = a.A == 1 ? a.H : a.H / a.H_kv;
    const int y = u % hpa;
    const focus_item_t it = a.items[a.order[u / hpa]];
    U.b = it.b;
    asg = it.a;
    U.h = a.A == 1 ? y : it.a * (a.H / a.H_kv) + y;
    kv = (U.h * a.H_kv) / a.H;
    U.prob = U.b * a.A + asg;
    const int rA = min(kHalf, it.rows), rB = it.rows - kHalf;
    const int kA = a.farlen_slot[static_cast<size_t>(U.prob) * a.n + it.row0 + rA - 1];
    const int kB = rB > 0 ? it.keys : 0;
    U.row0[0] = it.row0;
    U.nrows[0] = rA;
    U.row0[1] = it.row0 + kHalf;
    U.nrows[1] = rB;
    U.t0[0] = 0;
    U.t1[0] = (kA + kBN - 1) / kBN - 1;
    U.t0[1] = 0;
    U.t1[1] = (kB + kBN - 1) / kBN - 1;
    U.ybase = it.key0;
  } else {
    U.h = u % a.H;
    const int r = u / a.H;
    const int nqp = (a.n + kUnitRows - 1) / kUnitRows;
    const int qp = nqp - 1 - (r % nqp);          // longest units first
    U.b = r / nqp;
    kv = (U.h * a.H_kv) / a.H;
    asg = a.A == 1 ? 0 : kv;
    U.prob = U.b * a.A + asg;
    for (int x = 0; x < 2; ++x) {
      U.row0[x] = qp * kUnitRows + x * kHalf;
      U.nrows[x] = min(kHalf, a.n - U.row0[x]);
      if (U.nrows[x] <= 0) {
        U.t0[x] = 0;
        U.t1[x] = -1;
      } else {
        U.t0[x] = MODE == kModeDense ? 0 : max(0, U.row0[x] - a.w + 1) / kBN;
        U.t1[x] = (U.row0[x] + U.nrows[x] - 1) / kBN;
      }
    }
    U.ybase = 0;
  }
  U.zkv = U.b * a.H_kv + kv;
  U.zq = U.b * a.H + U.h;
  const bool a0 = active(U, 0), a1 = active(U, 1);
  U.T0 = a0 ? (a1 ? min(U.t0[0], U.t0[1]) : U.t0[0]) : U.t0[1];
  U.T1 = a0 ? (a1 ? max(U.t1[0], U.t1[1]) : U.t1[0]) : U.t1[1];
}

template <int D, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const AttnArgs a) {
  using Cfg = AttnCfg<D>;
  constexpr int kChunks = D / 64;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + Cfg::kQ;
  uint8_t* sKV = smem + Cfg::kRing;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kBar);
  uint64_t* q_full = bars + 0;     // [2] per half
  uint64_t* q_empty = bars + 2;    // [2]
  uint64_t* kv_full = bars + 4;    // [kKvSlots]
  uint64_t* kv_empty = bars + 4 + kKvSlots;
  uint64_t* s_full = bars + 4 + 2 * kKvSlots;    // [2] per half
  uint64_t* p_ready = s_full + 2;  // [2]
  uint64_t* o_final = s_full + 4;  // [2]
  uint64_t* o_free = s_full + 6;   // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_full + 8);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = warp_id(), lane = lane_id();
  const int n_units = unit_count<MODE>(a);
  if (threadIdx.x == 0) {
    for (int x = 0; x < 2; ++x) {
      mbar_init(&q_full[x], MODE == kModeGroup ? 32 : 1);
      mbar_init(&q_empty[x], 1);
      mbar_init(&s_full[x], 1);
      mbar_init(&p_ready[x], 128);
      mbar_init(&o_final[x], 1);
      mbar_init(&o_free[x], 128);
    }
    for (int k = 0; k < kKvSlots; ++k) {
      mbar_init(&kv_full[k], 1);
      mbar_init(&kv_empty[k], 1);
    }
    *abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  if (warp == 9) tmem_alloc(tmem_slot, Cfg::kTmemCols);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 8) {
    // warpgroup 2: one register budget for the load and MMA roles
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
    if (warp == 8) {
    // ---------------------------------------------------------- loads ---
    int c = 0;                 // K/V tiles walked
    int issued = 0;            // K/V loads issued (lane 0)
    int qn[2] = {0, 0};        // Q loads issued per half
    bool ok = true;
    const __nv_bfloat16* Qg = static_cast<const __nv_bfloat16*>(a.Q);
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      Unit U;
      decode_unit<MODE>(a, u, U);
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        if (!ok || !active(U, x)) continue;
        if (qn[x] > 0 && !warp_wait(&q_empty[x], (qn[x] - 1) & 1, abort, a.err)) { ok = false; break; }
        uint8_t* dstq = sQ + x * Cfg::kTile;
        if (MODE == kModeGroup) {
          // gather 128 rows through perm, four rows per lane, zero past the item
          for (int k = 0; k < kHalf / 32; ++k) {
            const int r = lane + 32 * k;
            const bool valid = r < U.nrows[x];
            const int pos = valid ? a.perm[static_cast<size_t>(U.prob) * a.n + U.row0[x] + r] : 0;
            const __nv_bfloat16* src = Qg + (static_cast<size_t>(U.zq) * a.n + pos) * D;
#pragma unroll
            for (int v = 0; v < D / 8; ++v)
              cp_async_16(dstq + (v >> 3) * Cfg::kChunk + r * 128 + (((v & 7) ^ (r & 7)) << 4),
                          src + v * 8, valid ? 16u : 0u);
          }
          cp_async_wait_all();
          fence_proxy_async_smem();
          mbar_arrive(&q_full[x]);
        } else if (lane == 0) {
          mbar_expect_tx(&q_full[x], Cfg::kTile);
#pragma unroll
          for (int ch = 0; ch < kChunks; ++ch)
            tma_load_3d(dstq + ch * Cfg::kChunk, &tm_q, &q_full[x], ch * 64, U.row0[x], U.zq);
        }
        ++qn[x];
      }
      if (!ok) break;
      if (lane == 0) {
        // load L = 2c (K of tile c) and 2c+1 (V of tile c) into slot L % kKvSlots
        for (int t = U.T0; t <= U.T1 && ok; ++t, ++c) {
          const int y = U.ybase + t * kBN;
#pragma unroll
          for (int kv = 0; kv < 2; ++kv) {
            const int L = 2 * c + kv, sl = L % kKvSlots, use = L / kKvSlots;
            if (use > 0 && !mbar_wait(&kv_empty[sl], (use - 1) & 1, abort, a.err)) { ok = false; break; }
            mbar_expect_tx(&kv_full[sl], Cfg::kTile);
#pragma unroll
            for (int ch = 0; ch < kChunks; ++ch)
              tma_load_3d(sKV + sl * Cfg::kTile + ch * Cfg::kChunk, kv ? &tm_v : &tm_k, &kv_full[sl],
                          ch * 64, y, U.zkv);
            ++issued;
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0) && !*abort;
      c = __shfl_sync(0xffffffffu, c, 0);
    }
    if (*abort && lane == 0) {
      // drain: TMA copies already issued must land before the CTA exits
      for (int L = max(0, issued - kKvSlots); L < issued; ++L) {
        const unsigned long long t0 = global_ns();
        while (!mbar_try_wait(&kv_full[L % kKvSlots], (L / kKvSlots) & 1) &&
               global_ns() - t0 < kWaitTimeoutNs) {}
      }
      if (MODE != kModeGroup) {
        for (int x = 0; x < 2; ++x) {
          if (qn[x] == 0) continue;
          const unsigned long long t0 = global_ns();
          while (!mbar_try_wait(&q_full[x], (qn[x] - 1) & 1) && global_ns() - t0 < kWaitTimeoutNs) {}
        }
      }
    }
    } else if (warp == 9) {
    // ----------------------------------------------------------- MMAs ---
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, kBN, false, false);
      constexpr uint32_t idPV = idesc_bf16_f32(128, D, false, true);
      const uint32_t q0 = smem_u32(sQ), r0 = smem_u32(sKV);
      int c = 0;                   // K/V tiles consumed
      int qn[2] = {0, 0};          // units per half
      int pv[2] = {0, 0};          // PV products issued per half
      bool ok = true;
      // descriptor low words: Q halves and ring slots as K-major operands
      // (LBO unused), ring slots as MN-major V operands (LBO = one 64-column slab)
      constexpr uint32_t dhi = sw128_desc_hi();
      const uint32_t qlo = sw128_desc_lo(q0, 16), klo = sw128_desc_lo(r0, 16);
      const uint32_t vlo = sw128_desc_lo(r0, Cfg::kChunk);
      auto issue_s = [&](int x, int st) {
        const uint32_t a0 = qlo + x * (Cfg::kTile >> 4), b0 = klo + st * (Cfg::kTile >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * Cfg::kChunk + (kk & 3) * 32) >> 4;
          mma_ss(tmem + 128 * x, desc_join(a0 + off, dhi), desc_join(b0 + off, dhi), idS, kk > 0);
        }
        mma_commit(&s_full[x]);
      };
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        Unit U;
        decode_unit<MODE>(a, u, U);
        bool first[2] = {true, true};
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (ok && active(U, x) && !mbar_wait(&q_full[x], qn[x] & 1, abort, a.err)) ok = false;
        }
        if (!ok) break;
        // first key tile: S products only
        if (!mbar_wait(&kv_full[(2 * c) % kKvSlots], ((2 * c) / kKvSlots) & 1, abort, a.err)) break;
        tc_fence_after();
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (!active_at(U, x, U.T0)) continue;
          issue_s(x, (2 * c) % kKvSlots);
          if (U.T0 == U.t1[x]) mma_commit(&q_empty[x]);
        }
        mma_commit(&kv_empty[(2 * c) % kKvSlots]);
        for (int t = U.T0; t <= U.T1 && ok; ++t, ++c) {
          const int st = (2 * c + 1) % kKvSlots;          // V of this tile
          const int stn = (2 * c + 2) % kKvSlots;         // K of the next tile
          const bool next = t < U.T1;
          if (!mbar_wait(&kv_full[st], ((2 * c + 1) / kKvSlots) & 1, abort, a.err)) { ok = false; break; }
          if (next && !mbar_wait(&kv_full[stn], ((2 * c + 2) / kKvSlots) & 1, abort, a.err)) { ok = false; break; }
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            if (!ok) continue;
            if (active_at(U, x, t)) {
              if (first[x] && qn[x] > 0 && !mbar_wait(&o_free[x], (qn[x] - 1) & 1, abort, a.err)) { ok = false; continue; }
              if (!mbar_wait(&p_ready[x], pv[x] & 1, abort, a.err)) { ok = false; continue; }
              tc_fence_after();
              const uint32_t vb = vlo + st * (Cfg::kTile >> 4);
#pragma unroll
              for (int kk = 0; kk < kBN / 16; ++kk)
                mma_ts(tmem + 256 + 128 * x, tmem + 128 * x + kk * 8,
                       desc_join(vb + kk * ((16 * 128) >> 4), dhi), idPV, (!first[x]) || kk > 0);
              ++pv[x];
              first[x] = false;
              if (t == U.t1[x]) mma_commit(&o_final[x]);
            }
            if (next && active_at(U, x, t + 1)) {
              tc_fence_after();
              issue_s(x, stn);
              if (t + 1 == U.t1[x]) mma_commit(&q_empty[x]);
            }
          }
          if (!ok) break;
          mma_commit(&kv_empty[st]);
          if (next) mma_commit(&kv_empty[stn]);
        }
#pragma unroll
        for (int x = 0; x < 2; ++x)
          if (active(U, x)) ++qn[x];
      }
    }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
    // -------------------------------------------------------- softmax ---
    const int x = warp >> 2;              // half served by this warpgroup
    const int qw = warp & 3;              // TMEM lane quarter
    const int r = qw * 32 + lane;         // row within the half
    const uint32_t lane_base = static_cast<uint32_t>(qw * 32) << 16;
    const uint32_t tS = tmem + lane_base + 128 * x;
    const uint32_t tO = tmem + lane_base + 256 + 128 * x;
    const float sl2 = a.scale_log2;
    constexpr float kLn2 = 0.6931471805599453f;
    constexpr float kLog2e = 1.4426950408889634f;
    int sn = 0, un = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      Unit U;
      decode_unit<MODE>(a, u, U);
      const int my_t0 = x ? U.t0[1] : U.t0[0];
      const int my_t1 = x ? U.t1[1] : U.t1[0];
      const int my_row0 = x ? U.row0[1] : U.row0[0];
      const int my_nrows = x ? U.nrows[1] : U.nrows[0];
      if (my_t1 < my_t0) continue;
      const bool valid = r < my_nrows;
      int pos = -1, lo = 1, hi = 0;
      if (MODE == kModeGroup) {
        if (valid) {
          const size_t sidx = static_cast<size_t>(U.prob) * a.n + my_row0 + r;
          pos = a.perm[sidx];
          lo = 0;
          hi = a.farlen_slot[sidx] - 1;
        }
      } else if (valid) {
        pos = my_row0 + r;
        lo = MODE == kModeDense ? 0 : pos - a.w + 1;
        hi = pos;
      }
      float m_run = -INFINITY, l = 0.f;
      for (int t = my_t0; t <= my_t1; ++t) {
        const int j0 = t * kBN;
        if (!warp_wait(&s_full[x], sn & 1, abort, a.err)) { ok = false; break; }
        ++sn;
        tc_fence_after();
        // S row: four 32-column loads in flight, one wait
        uint32_t su[kBN];
#pragma unroll
        for (int c = 0; c < kBN; c += 32)
          tmem_ld32(tS + c, *reinterpret_cast<uint32_t(*)[32]>(&su[c]));
        tmem_wait_ld();
        const bool full = j0 >= lo && j0 + kBN - 1 <= hi;
        if (!full) {
#pragma unroll
          for (int c = 0; c < kBN; ++c)
            if (j0 + c < lo || j0 + c > hi) su[c] = __float_as_uint(-INFINITY);
        }
        // row max: eight independent chains, then a tree
        float m8[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) m8[j] = __uint_as_float(su[j]);
#pragma unroll
        for (int c = 8; c < kBN; c += 8)
#pragma unroll
          for (int j = 0; j < 8; ++j) m8[j] = fmaxf(m8[j], __uint_as_float(su[c + j]));
        const float mt = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                               fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
        const float m_new = fmaxf(m_run, mt * sl2);
        const bool need = m_run != -INFINITY && m_new > m_run + kRescaleThreshold;
        if (m_run == -INFINITY) m_run = m_new;      // nothing accumulated yet for this row
        if (__any_sync(0xffffffffu, need)) {
          // S_X(t) landed after PV_X(t-1): O_X is complete up to tile t-1
          const float alpha = need ? ex2f(m_run - m_new) : 1.f;
          uint32_t rr[32];
#pragma unroll
          for (int c = 0; c < D; c += 32) {
            tmem_ld32(tO + c, rr);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * alpha);
            tmem_st32(tO + c, rr);
          }
          if (need) {
            l *= alpha;
            m_run = m_new;
          }
        }
        const float mu = m_run == -INFINITY ? 0.f : m_run;
        // p = 2^(s*scale*log2e - m): scale-and-shift in packed pairs, exp2 per
        // element (MUFU, or the FMA-pipe polynomial for part of a fully kept
        // tile), four packed partial sums; P is written back as bf16 over the
        // first 64 columns of S, which this thread has already read
        const uint64_t sc2 = f2_pack(sl2, sl2), nm2 = f2_pack(-mu, -mu);
        uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            const int col = 64 * h2 + c;
            float t0, t1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(su[col]), __uint_as_float(su[col + 1])), sc2, nm2), t0, t1);
            float p0, p1;
            if ((col & 7) < FOCUS_EXP_POLY_PER8 && full) {
              p0 = exp2_poly(t0);
              p1 = exp2_poly(t1);
            } else {
              p0 = ex2f(t0);
              p1 = ex2f(t1);
            }
            acc[(c >> 1) & 3] = f2_add(acc[(c >> 1) & 3], f2_pack(p0, p1));
            pk[c / 2] = pack_bf16x2(p0, p1);
          }
          tmem_st32(tS + 32 * h2, pk);
        }
        {
          const uint64_t s2 = f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3]));
          float s0, s1;
          f2_unpack(s2, s0, s1);
          l += s0 + s1;
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&p_ready[x]);
      }
      if (!ok) break;

      // ---------------------------------------------------- epilogue ---
      if (!warp_wait(&o_final[x], un & 1, abort, a.err)) { ok = false; break; }
      tc_fence_after();
      const size_t qrow = static_cast<size_t>(U.zq) * a.n;
      float c1 = l > 0.f ? 1.f / l : 0.f, c2 = 0.f;
      float lse2 = m_run + log2f(l);
      bool far = false;
      const size_t orow = (qrow + (valid ? pos : 0)) * D;
      const __nv_bfloat16* Of = static_cast<const __nv_bfloat16*>(a.O_far);
      if (MODE == kModeLocal && valid) {
        far = a.farlen_tok[static_cast<size_t>(U.prob) * a.n + pos] > 0;
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
        tmem_ld32(tO + c, rr);
        tmem_wait_ld();
        if (write) {
          float f[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(rr[e]) * c1;
          if (far) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const uint4 g4 = *reinterpret_cast<const uint4*>(Of + orow + c + v * 8);
              const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&g4);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 g = __bfloat1622float2(g2[e]);
                f[v * 8 + 2 * e] = fmaf(g.x, c2, f[v * 8 + 2 * e]);
                f[v * 8 + 2 * e + 1] = fmaf(g.y, c2, f[v * 8 + 2 * e + 1]);
              }
            }
          }
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 o4;
            o4.x = pack_bf16x2(f[v * 8 + 0], f[v * 8 + 1]);
            o4.y = pack_bf16x2(f[v * 8 + 2], f[v * 8 + 3]);
            o4.z = pack_bf16x2(f[v * 8 + 4], f[v * 8 + 5]);
            o4.w = pack_bf16x2(f[v * 8 + 6], f[v * 8 + 7]);
            *reinterpret_cast<uint4*>(dst + orow + c + v * 8) = o4;
          }
        }
      }
      if (write) {
        if (MODE == kModeGroup) a.lse_far[qrow + pos] = lse2 * kLn2;
        else if (a.lse) a.lse[qrow + pos] = lse2 * kLn2;
      }
      tc_fence_before();
      mbar_arrive(&o_free[x]);
      ++un;
    }
  }

  __syncwarp();          // lanes of warps 8 and 9 reconverge before the CTA barrier
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
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
cudaError_t launch_d(const AttnArgs& a, const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                     const CUtensorMap* tm_v, int mode, int max_items, int num_sms, cudaStream_t st) {
  using Cfg = AttnCfg<D>;
  long long units;
  if (mode == kModeGroup) {
    const int hpa = a.A == 1 ? a.H : a.H / a.H_kv;
    units = static_cast<long long>(max_items) * hpa;
  } else {
    units = static_cast<long long>(a.B) * a.H * ((a.n + kUnitRows - 1) / kUnitRows);
  }
  if (units == 0) return cudaSuccess;
  const unsigned grid = static_cast<unsigned>(units < num_sms ? units : num_sms);
  if (mode == kModeGroup)
    attn_tc_kernel<D, kModeGroup><<<grid, kThreads, Cfg::kSmem, st>>>(*tm_q, *tm_k, *tm_v, a);
  else if (mode == kModeLocal)
    attn_tc_kernel<D, kModeLocal><<<grid, kThreads, Cfg::kSmem, st>>>(*tm_q, *tm_k, *tm_v, a);
  else
    attn_tc_kernel<D, kModeDense><<<grid, kThreads, Cfg::kSmem, st>>>(*tm_q, *tm_k, *tm_v, a);
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

cudaError_t launch_attn_tc_bf16(const AttnArgs& a, const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                const CUtensorMap* tm_v, int d, int mode, int max_items, int num_sms,
                                cudaStream_t st) {
  if (d == 64) return launch_d<64>(a, tm_q, tm_k, tm_v, mode, max_items, num_sms, st);
  if (d == 128) return launch_d<128>(a, tm_q, tm_k, tm_v, mode, max_items, num_sms, st);
  return cudaErrorInvalidValue;
}

cudaError_t setup_attn_kernels() {
  cudaError_t e = set_smem<64>();
  if (e != cudaSuccess) return e;
  return set_smem<128>();
}

}  // namespace focus
