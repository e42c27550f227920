// Backward of Focus attention on the tcgen05 tensor cores (bf16 tensors, fp32
// accumulate): the same gradients as attn_bwd.cu ("Why Attend to Everything?
// Focus is the Key", section 2.1; "Focus: Learning Which Attention Pairs
// Matter", section 3.1), with every d-long product an MMA.
//
// Two kernels, each in a group form (far pairs, rows and keys in the index's
// sorted order, read as TMA tiles from copies of Q, dO, K, V (and LSE, Delta)
// sorted by the index once per call) and a window form (natural order, TMA
// tiles); one CTA per 128-row unit:
//   dQ   rows = 128 queries, streamed = 128-key tiles of the kept keys:
//          S = Q K^T, dP = dO V^T               (SS, TMEM fp32)
//          dS = P (dP - Delta), P = exp(S scale - LSE)   (CUDA cores -> TMEM bf16)
//          dQ += dS K                           (TS, K as the MN-major operand)
//   dKV  rows = 128 keys, streamed = 128-query tiles of the queries that keep
//        them, for every query head of the key/value head:
//          S^T = K Q^T, dP^T = V dO^T           (SS)
//          P^T, dS^T                            (CUDA cores -> TMEM bf16)
//          dV += P^T dO, dK += dS^T Q           (TS)
// TMEM (512 columns): S at 0, dP at 128 (the bf16 P^T / dS^T overwrite their
// first 64 columns once read), accumulators at 256 (and 256 + d).  One tile is
// in flight at a time; the next tile's operands stream in through a 2-slot TMA
// ring meanwhile.  Warps 0-7 do the elementwise work, two per TMEM lane
// quadrant, each on half of the row's columns: both halves read their fp32
// columns, meet at an mbarrier, and only then write the bf16 pairs over the
// first half of the fp32 columns.  Warp 8 loads, warp 9 owns TMEM and issues
// the MMAs.  Every wait is bounded; on a timeout the CTA raises the error bit,
// drains and exits.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace focus {
namespace {

constexpr int kT = 128;
constexpr int kEwWarps = 8;
constexpr int kWarpLd = 8;
constexpr int kWarpMma = 9;
constexpr int kThreads = 320;
constexpr float kLog2e = 1.4426950408889634f;

enum : int { kDqGroup = 0, kDqLocal = 1, kDkvGroup = 2, kDkvLocal = 3 };

template <int D>
struct BCfg {
  static constexpr int kChunk = 128 * 128;   // 128 rows x 64 bf16, one swizzle slab
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kF0 = 0;              // fixed operands of the unit
  static constexpr int kF1 = kTile;
  static constexpr int kR = 2 * kTile;       // ring: 2 slots x (R0, R1)
  static constexpr int kCol = kR + 4 * kTile;              // [2 slots][lse2, delta][128] fp32
  static constexpr int kBar = kCol + 2 * 2 * 128 * 4;
  static constexpr int kMisc = kBar + 256;
  static constexpr int kBytes = kMisc + 64;
  static constexpr int kSmem = kBytes + 1024;             // + slack to align the base to 1024
  static constexpr uint32_t kS = 0, kDP = 128, kA0 = 256, kA1 = 256 + D;
};
static_assert(BCfg<128>::kSmem <= 227 * 1024, "backward shared memory above 227 KB");

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void warp_arrive(uint64_t* bar, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          int* err) {
  const bool ok = mbar_wait(bar, parity, abort, err);
  return __all_sync(0xffffffffu, ok);
}

struct BUnit {
  bool valid;
  int b, kv, h, prob, zq, zkv;
  int row0, nrows;      // the unit's rows: query (dQ) or key (dKV) slots / tokens
  int key0, nkeys;      // dQ group: key slots [key0, key0 + nkeys); dQ local: first key token
  int ntile;            // streamed tiles per query head
  int heads;            // query heads walked (dKV: H / H_kv; dQ: 1)
};

template <int KIND>
__device__ __forceinline__ BUnit decode(const BwdArgs& a, int u) {
  BUnit U{};
  U.valid = true;
  U.heads = 1;
  if (KIND == kDqGroup) {
    const int hpa = a.A == 1 ? a.H : a.H / a.H_kv;
    const int y = u % hpa, io = u / hpa;
    if (io >= *a.n_items) {
      U.valid = false;
      return U;
    }
    const focus_item_t it = a.items[a.order[io]];
    U.b = it.b;
    U.h = a.A == 1 ? y : it.a * (a.H / a.H_kv) + y;
    U.kv = (U.h * a.H_kv) / a.H;
    U.prob = it.b * a.A + it.a;
    U.row0 = it.row0;
    U.nrows = it.rows;
    U.key0 = it.key0;
    U.nkeys = it.keys;
    U.ntile = (it.keys + kT - 1) / kT;
  } else if (KIND == kDqLocal) {
    U.h = u % a.H;
    const int r = u / a.H;
    const int nqt = (a.n + kT - 1) / kT;
    const int qt = nqt - 1 - (r % nqt);
    U.b = r / nqt;
    U.kv = (U.h * a.H_kv) / a.H;
    U.prob = U.b * a.A + (a.A == 1 ? 0 : U.kv);
    U.row0 = qt * kT;
    U.nrows = min(kT, a.n - U.row0);
    const int kt0 = max(0, U.row0 - a.w + 1) / kT;
    U.key0 = kt0 * kT;
    U.ntile = (U.row0 + U.nrows - 1) / kT - kt0 + 1;
  } else {
    const int nkt = (a.n + kT - 1) / kT;
    const int kt = u % nkt, r = u / nkt;
    U.kv = r % a.H_kv;
    U.b = r / a.H_kv;
    U.h = U.kv * (a.H / a.H_kv);
    U.prob = U.b * a.A + (a.A == 1 ? 0 : U.kv);
    U.row0 = kt * kT;
    U.nrows = min(kT, a.n - U.row0);
    U.heads = a.H / a.H_kv;
  }
  U.zq = U.b * a.H + U.h;
  U.zkv = U.b * a.H_kv + U.kv;
  return U;
}

template <int D, int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const BwdArgs a) {
  using Cfg = BCfg<D>;
  constexpr int kChunks = D / 64;
  constexpr bool kDq = KIND == kDqGroup || KIND == kDqLocal;
  constexpr bool kGroup = KIND == kDqGroup || KIND == kDkvGroup;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kBar);
  uint64_t* fixed_full = bars + 0;
  uint64_t* ring_full = bars + 1;     // [2]
  uint64_t* ring_empty = bars + 3;    // [2]
  uint64_t* sp_full = bars + 5;
  uint64_t* ew_done = bars + 6;
  uint64_t* acc_done = bars + 7;
  uint64_t* mma_done = bars + 8;
  uint64_t* col_full = bars + 9;      // [2] dKV: the slot's query LSE / Delta are in shared memory
  uint64_t* read_done = bars + 11;    // every elementwise warp has read this tile's fp32 S and dP
  int* misc = reinterpret_cast<int*>(smem + Cfg::kMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 0);
  volatile int* abort = misc + 1;
  int* range = misc + 2;              // dKV: walked query range [range[0], range[1]]
  float* colbuf = reinterpret_cast<float*>(smem + Cfg::kCol);

  const int warp = warp_id(), lane = lane_id();
  const BUnit U = decode<KIND>(a, static_cast<int>(blockIdx.x));
  if (!U.valid) return;
  const size_t pn = static_cast<size_t>(U.prob) * a.n;

  if (threadIdx.x == 0) {
    mbar_init(fixed_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&ring_full[s], 1);
      mbar_init(&ring_empty[s], 1);
    }
    mbar_init(sp_full, 1);
    mbar_init(ew_done, kEwWarps);
    mbar_init(read_done, kEwWarps);
    mbar_init(acc_done, 1);
    mbar_init(mma_done, 1);
    mbar_init(&col_full[0], 32);
    mbar_init(&col_full[1], 32);
    *abort = 0;
    range[0] = 0x7fffffff;
    range[1] = -1;
    fence_mbar_init();
  }
  if (warp == kWarpMma) tmem_alloc(tmem_slot, 512);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // ---- per-row bookkeeping of the elementwise threads (row = TMEM lane) ----
  const int r = (warp & 3) * 32 + lane;
  const int half = (warp >> 2) & 1;   // elementwise: which half of the columns
  const bool row_ok = warp < kEwWarps && r < U.nrows;
  int rpos = -1;        // token of the row
  int klo = 1, khi = 0; // kept streamed indices of the row (inclusive), in the walked order
  if (warp < kEwWarps && row_ok) {
    if (KIND == kDqGroup) {
      rpos = a.perm[pn + U.row0 + r];
      klo = 0;
      khi = a.farlen_slot[pn + U.row0 + r] - 1;           // prefix index
    } else if (KIND == kDqLocal) {
      rpos = U.row0 + r;
      klo = rpos - a.w + 1;
      khi = rpos;                                         // key tokens
    } else if (KIND == kDkvGroup) {
      const int u = U.row0 + r;
      rpos = a.perm[pn + u];
      const int32_t* off = a.offsets + static_cast<size_t>(U.prob) * (a.groups + 1);
      int glo = 0, ghi = a.groups;
      while (ghi - glo > 1) {
        const int mid = (glo + ghi) >> 1;
        if (off[mid] <= u) glo = mid; else ghi = mid;
      }
      const int gend = off[glo + 1];
      const int target = rpos + a.w;
      int s0 = u + 1, s1 = gend;
      while (s0 < s1) {
        const int mid = (s0 + s1) >> 1;
        if (a.perm[pn + mid] < target) s0 = mid + 1; else s1 = mid;
      }
      klo = s0;
      khi = gend - 1;                                     // query slots
    } else {
      rpos = U.row0 + r;
      klo = rpos;
      khi = min(a.n - 1, rpos + a.w - 1);                 // query tokens
    }
  }
  if (!kDq) {
    if (row_ok && klo <= khi) {
      atomicMin(&range[0], klo);
      atomicMax(&range[1], khi);
    }
    __syncthreads();
  }
  int wlo = 0, ntile = U.ntile;
  if (!kDq) {
    wlo = range[0];
    const int whi = range[1];
    ntile = whi >= wlo ? (whi - wlo) / kT + 1 : 0;
  }
  const int ntot = ntile * U.heads;

  if (warp == kWarpLd) {
    // ------------------------------------------------------------ loads ---
    bool ok = true;
    int issued = 0;
    if (ntot > 0) {
      // fixed operands: dQ -> (Q, dO) rows of the unit; dKV -> (K, V) rows
      // (group kinds: rows of the sorted copies, so one tile either way)
      if (lane == 0) {
        mbar_expect_tx(fixed_full, 2 * Cfg::kTile);
#pragma unroll
        for (int ch = 0; ch < kChunks; ++ch) {
          tma_load_3d(smem + Cfg::kF0 + ch * Cfg::kChunk, kDq ? &tm_q : &tm_k, fixed_full, ch * 64, U.row0,
                      kDq ? U.zq : U.zkv);
          tma_load_3d(smem + Cfg::kF1 + ch * Cfg::kChunk, kDq ? &tm_do : &tm_v, fixed_full, ch * 64, U.row0,
                      kDq ? U.zq : U.zkv);
        }
      }
      for (int it = 0; it < ntot && ok; ++it) {
        const int sl = it & 1, use = it >> 1;
        if (use > 0 && !mbar_wait_nap(&ring_empty[sl], (use - 1) & 1, abort, a.err)) ok = false;
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        const int t = it % ntile, hh = it / ntile;
        const int zq = U.b * a.H + U.h + hh;
        uint8_t* r0 = smem + Cfg::kR + sl * 2 * Cfg::kTile;
        uint8_t* r1 = r0 + Cfg::kTile;
        // dQ: key slots (group) or tokens from key0 + t*128; dKV: query slots or
        // tokens from wlo + t*128 (rows past a group's run are masked out)
        if (lane == 0) {
          mbar_expect_tx(&ring_full[sl], 2 * Cfg::kTile);
          const int y = (kDq ? U.key0 : wlo) + t * kT;
#pragma unroll
          for (int ch = 0; ch < kChunks; ++ch) {
            tma_load_3d(r0 + ch * Cfg::kChunk, kDq ? &tm_k : &tm_q, &ring_full[sl], ch * 64, y, kDq ? U.zkv : zq);
            tma_load_3d(r1 + ch * Cfg::kChunk, kDq ? &tm_v : &tm_do, &ring_full[sl], ch * 64, y, kDq ? U.zkv : zq);
          }
        }
        if (!kDq) {
          // the tile's query columns: LSE (log2 units) and Delta for head h + hh;
          // the slot is free (ring_empty above), and each lane's arrival
          // publishes its four entries
          float* cb = colbuf + sl * 256;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int c = 4 * lane + j;
            const int q = wlo + t * kT + c;
            float l2 = 0.f, dl = 0.f;
            if (q < a.n) {
              // group: the sorted copies are indexed by slot
              const size_t qi = static_cast<size_t>(zq) * a.n + q;
              l2 = (kGroup ? a.lse_sorted : a.lse)[qi] * kLog2e;
              dl = (kGroup ? a.delta_sorted : a.delta)[qi];
            }
            cb[c] = l2;
            cb[128 + c] = dl;
          }
          mbar_arrive(&col_full[sl]);
        }
        ++issued;
      }
      if ((*abort || !ok) && lane == 0) {
        // copies already issued must land before the CTA exits
        const unsigned long long t0 = global_ns();
        while (!mbar_try_wait(fixed_full, 0) && global_ns() - t0 < kWaitTimeoutNs) {}
        for (int it = max(0, issued - 2); it < issued; ++it) {
          const unsigned long long t1 = global_ns();
          while (!mbar_try_wait(&ring_full[it & 1], (it >> 1) & 1) && global_ns() - t1 < kWaitTimeoutNs) {}
        }
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------- MMAs ---
    if (lane == 0 && ntot > 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, kT, false, false);
      constexpr uint32_t idAcc = idesc_bf16_f32(128, D, false, true);
      constexpr uint32_t dhi = sw128_desc_hi();
      const uint32_t f0 = sw128_desc_lo(smem_u32(smem + Cfg::kF0), 16);
      const uint32_t f1 = sw128_desc_lo(smem_u32(smem + Cfg::kF1), 16);
      bool ok = mbar_wait_nap(fixed_full, 0, abort, a.err);
      for (int it = 0; it < ntot && ok; ++it) {
        const int sl = it & 1;
        if (!mbar_wait_nap(&ring_full[sl], (it >> 1) & 1, abort, a.err)) { ok = false; break; }
        if (it > 0 && !mbar_wait_nap(acc_done, (it - 1) & 1, abort, a.err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t rb = smem_u32(smem + Cfg::kR + sl * 2 * Cfg::kTile);
        const uint32_t r0k = sw128_desc_lo(rb, 16), r1k = sw128_desc_lo(rb + Cfg::kTile, 16);
        // S = F0 R0^T, dP = F1 R1^T (both operands K-major over d)
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * Cfg::kChunk + (kk & 3) * 32) >> 4;
          mma_ss(tmem + Cfg::kS, desc_join(f0 + off, dhi), desc_join(r0k + off, dhi), idS, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * Cfg::kChunk + (kk & 3) * 32) >> 4;
          mma_ss(tmem + Cfg::kDP, desc_join(f1 + off, dhi), desc_join(r1k + off, dhi), idS, kk > 0);
        }
        mma_commit(sp_full);
        if (!mbar_wait_nap(ew_done, it & 1, abort, a.err)) { ok = false; break; }
        tc_fence_after();
        // accumulators: the streamed tiles as MN-major operands (reduction over the tile's rows)
        const uint32_t r0m = sw128_desc_lo(rb, Cfg::kChunk), r1m = sw128_desc_lo(rb + Cfg::kTile, Cfg::kChunk);
        if (kDq) {
#pragma unroll
          for (int kk = 0; kk < kT / 16; ++kk)
            mma_ts(tmem + Cfg::kA0, tmem + Cfg::kDP + kk * 8, desc_join(r0m + kk * ((16 * 128) >> 4), dhi), idAcc,
                   it > 0 || kk > 0);
        } else {
#pragma unroll
          for (int kk = 0; kk < kT / 16; ++kk)
            mma_ts(tmem + Cfg::kA0, tmem + Cfg::kS + kk * 8, desc_join(r1m + kk * ((16 * 128) >> 4), dhi), idAcc,
                   it > 0 || kk > 0);
#pragma unroll
          for (int kk = 0; kk < kT / 16; ++kk)
            mma_ts(tmem + Cfg::kA1, tmem + Cfg::kDP + kk * 8, desc_join(r0m + kk * ((16 * 128) >> 4), dhi), idAcc,
                   it > 0 || kk > 0);
        }
        mma_commit(acc_done);
        mma_commit(&ring_empty[sl]);
      }
      // every MMA issued above has finished before TMEM is released
      mma_commit(mma_done);
      const unsigned long long t0 = global_ns();
      while (!mbar_try_wait(mma_done, 0) && global_ns() - t0 < kWaitTimeoutNs) {}
    }
  } else {
    // ------------------------------------------------------ elementwise ---
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float sl2 = a.scale_log2;
    float lse2 = 0.f, dlt = 0.f;
    if (kDq && row_ok) {
      const size_t qi = static_cast<size_t>(U.zq) * a.n + rpos;
      lse2 = a.lse[qi] * kLog2e;
      dlt = a.delta[qi];
    }
    bool ok = true;
    for (int it = 0; it < ntot && ok; ++it) {
      const int t = it % ntile;
      const float* cb = colbuf + (it & 1) * 256;  // [lse2 x128, delta x128] of this tile's queries
      if (!kDq && !warp_wait(&col_full[it & 1], (it >> 1) & 1, abort, a.err)) { ok = false; break; }
      if (!warp_wait(sp_full, it & 1, abort, a.err)) { ok = false; break; }
      tc_fence_after();
      // this half's 64 columns of S and dP, all read before anyone writes
      uint32_t sv[64], dv[64];
      tmem_ld32(tmem + lane_base + Cfg::kS + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
      tmem_ld32(tmem + lane_base + Cfg::kS + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
      tmem_ld32(tmem + lane_base + Cfg::kDP + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&dv[0]));
      tmem_ld32(tmem + lane_base + Cfg::kDP + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&dv[32]));
      tmem_wait_ld();
      tc_fence_before();
      warp_arrive(read_done, lane);
      if (!warp_wait(read_done, it & 1, abort, a.err)) { ok = false; break; }
      tc_fence_after();
      uint32_t pp[32], dd[32];
      const int base_idx = (kDq ? (KIND == kDqGroup ? 0 : U.key0) : wlo) + t * kT + half * 64;
#pragma unroll
      for (int e = 0; e < 64; e += 2) {
        float p2[2], d2[2];
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2) {
          const int col = half * 64 + e + q2;
          const int idx = base_idx + e + q2;
          const bool keep = row_ok && idx >= klo && idx <= khi;
          const float l2 = kDq ? lse2 : cb[col];
          const float dl = kDq ? dlt : cb[128 + col];
          const float p = keep ? ex2f(__uint_as_float(sv[e + q2]) * sl2 - l2) : 0.f;
          p2[q2] = p;
          d2[q2] = p * (__uint_as_float(dv[e + q2]) - dl);
        }
        pp[e / 2] = pack_bf16x2(p2[0], p2[1]);
        dd[e / 2] = pack_bf16x2(d2[0], d2[1]);
      }
      // the half's 64 bf16 values take packed columns 32*half .. 32*half + 31
      tmem_st32(tmem + lane_base + Cfg::kDP + half * 32, dd);
      if (!kDq) tmem_st32(tmem + lane_base + Cfg::kS + half * 32, pp);
      tmem_wait_st();
      tc_fence_before();
      warp_arrive(ew_done, lane);
    }
    // epilogue: the accumulators once the last tile's MMAs are done
    const bool have = ok && ntot > 0;
    if (have && !warp_wait(acc_done, (ntot - 1) & 1, abort, a.err)) ok = false;
    if (ok) {
      tc_fence_after();
      const size_t orow = static_cast<size_t>(kDq ? U.zq : U.zkv) * a.n + (rpos >= 0 ? rpos : 0);
      // this half's accumulator columns: [half * D/2, (half + 1) * D/2)
#pragma unroll 1
      for (int c = half * (D / 64); c < (half + 1) * (D / 64); ++c) {
        uint32_t x0[32], x1[32];
        if (have) {
          tmem_ld32(tmem + lane_base + Cfg::kA0 + c * 32, x0);
          if (!kDq) tmem_ld32(tmem + lane_base + Cfg::kA1 + c * 32, x1);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) x0[e] = x1[e] = 0u;
        }
        if (!row_ok) continue;
        const size_t o = orow * D + c * 32;
        if (KIND == kDqGroup) {
          float4* dst = reinterpret_cast<float4*>(a.dq_far + o);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            dst[v] = make_float4(__uint_as_float(x0[4 * v]) * a.scale, __uint_as_float(x0[4 * v + 1]) * a.scale,
                                 __uint_as_float(x0[4 * v + 2]) * a.scale, __uint_as_float(x0[4 * v + 3]) * a.scale);
        } else if (KIND == kDqLocal) {
          const bool far = a.farlen_tok[pn + rpos] > 0;
          const float4* fq = reinterpret_cast<const float4*>(a.dq_far + o);
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.dQ) + o);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            float f[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(x0[8 * v + e]) * a.scale;
            if (far) {
              const float4 g0 = fq[2 * v], g1 = fq[2 * v + 1];
              f[0] += g0.x; f[1] += g0.y; f[2] += g0.z; f[3] += g0.w;
              f[4] += g1.x; f[5] += g1.y; f[6] += g1.z; f[7] += g1.w;
            }
            dst[v] = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                                pack_bf16x2(f[6], f[7]));
          }
        } else if (KIND == kDkvGroup) {
          float4* dvd = reinterpret_cast<float4*>(a.dv_far + o);
          float4* dkd = reinterpret_cast<float4*>(a.dk_far + o);
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            dvd[v] = make_float4(__uint_as_float(x0[4 * v]), __uint_as_float(x0[4 * v + 1]),
                                 __uint_as_float(x0[4 * v + 2]), __uint_as_float(x0[4 * v + 3]));
            dkd[v] = make_float4(__uint_as_float(x1[4 * v]) * a.scale, __uint_as_float(x1[4 * v + 1]) * a.scale,
                                 __uint_as_float(x1[4 * v + 2]) * a.scale, __uint_as_float(x1[4 * v + 3]) * a.scale);
          }
        } else {
          const float4* fv = reinterpret_cast<const float4*>(a.dv_far + o);
          const float4* fk = reinterpret_cast<const float4*>(a.dk_far + o);
          uint4* dvd = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.dV) + o);
          uint4* dkd = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.dK) + o);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const float4 v0 = fv[2 * v], v1 = fv[2 * v + 1], k0 = fk[2 * v], k1 = fk[2 * v + 1];
            const float gv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
            const float gk[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
            float fvv[8], fkk[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              fvv[e] = __uint_as_float(x0[8 * v + e]) + gv[e];
              fkk[e] = __uint_as_float(x1[8 * v + e]) * a.scale + gk[e];
            }
            dvd[v] = make_uint4(pack_bf16x2(fvv[0], fvv[1]), pack_bf16x2(fvv[2], fvv[3]),
                                pack_bf16x2(fvv[4], fvv[5]), pack_bf16x2(fvv[6], fvv[7]));
            dkd[v] = make_uint4(pack_bf16x2(fkk[0], fkk[1]), pack_bf16x2(fkk[2], fkk[3]),
                                pack_bf16x2(fkk[4], fkk[5]), pack_bf16x2(fkk[6], fkk[7]));
          }
        }
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// dQ kernels, persistent: one CTA per SM walks the units in snake order (a
// longest-first list for the group kind) and keeps two tiles in flight.  dS
// goes to its own TMEM double buffer (columns 384 + 64 * (tile & 1)), so the
// next tile's S and dP products run as soon as the elementwise warps have
// read this tile's fp32 S and dP, and the tensor pipe issues, per tile,
//   S(g), dP(g)  then  dQ += dS(g - 1) K(g - 1)
// K tiles sit in a 3-slot ring (freed by the dQ product two steps later), V
// tiles in a 2-slot ring (freed by the dP product), the unit's Q and dO rows
// in one fixed pair of tiles that the next unit's rows replace once the last
// S and dP products of the unit are done.
template <int D>
struct DqCfg {
  static constexpr int kChunk = 128 * 128;   // 128 rows x 64 bf16, one swizzle slab
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kKSlots = 3, kVSlots = 2;
  static constexpr int kF0 = 0;              // Q rows of the unit
  static constexpr int kF1 = kTile;          // dO rows of the unit
  static constexpr int kK = 2 * kTile;
  static constexpr int kV = kK + kKSlots * kTile;
  static constexpr int kBar = kV + kVSlots * kTile;
  static constexpr int kMisc = kBar + 256;
  static constexpr int kBytes = kMisc + 64;
  static constexpr int kSmem = kBytes + 1024;
  static constexpr uint32_t kS = 0, kDP = 128, kA = 256, kDS = 384;
};
static_assert(DqCfg<128>::kSmem <= 227 * 1024, "dQ shared memory above 227 KB");

// Unit k of this CTA in snake order over n_units (-1: past the end, -2: none this round).
__device__ __forceinline__ int bwd_snake(int k, int n_units) {
  const int G = gridDim.x, base = k * G;
  if (base >= n_units) return -1;
  const int u = base + ((k & 1) ? G - 1 - static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x));
  return u < n_units ? u : -2;
}

template <int D, int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const BwdArgs a) {
  using Cfg = DqCfg<D>;
  constexpr int kChunks = D / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kBar);
  uint64_t* fixed_full = bars + 0;
  uint64_t* fixed_empty = bars + 1;
  uint64_t* k_full = bars + 2;        // [3]
  uint64_t* k_empty = bars + 5;       // [3]
  uint64_t* v_full = bars + 8;        // [2]
  uint64_t* v_empty = bars + 10;      // [2]
  uint64_t* sp_full = bars + 12;
  uint64_t* read_done = bars + 13;    // every elementwise warp has read the tile's S and dP
  uint64_t* ew_done = bars + 14;      // [2] the tile's dS is in TMEM
  uint64_t* acc_full = bars + 16;     // the unit's dQ is complete
  uint64_t* mma_done = bars + 17;
  int* misc = reinterpret_cast<int*>(smem + Cfg::kMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 0);
  volatile int* abort = misc + 1;

  const int warp = warp_id(), lane = lane_id();
  const int n_units = KIND == kDqGroup ? *a.n_items * (a.A == 1 ? a.H : a.H / a.H_kv)
                                       : a.B * a.H * ((a.n + kT - 1) / kT);

  if (threadIdx.x == 0) {
    mbar_init(fixed_full, 1);
    mbar_init(fixed_empty, 1);
    for (int s = 0; s < Cfg::kKSlots; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < Cfg::kVSlots; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    mbar_init(sp_full, 1);
    mbar_init(read_done, kEwWarps);
    mbar_init(&ew_done[0], kEwWarps);
    mbar_init(&ew_done[1], kEwWarps);
    mbar_init(acc_full, 1);
    mbar_init(mma_done, 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) tmem_alloc(tmem_slot, 512);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kWarpLd) {
    // ------------------------------------------------------------ loads ---
    bool ok = true;
    int g = 0, uf = 0;
    for (int k = 0; ok; ++k) {
      const int u = bwd_snake(k, n_units);
      if (u == -1) break;
      if (u < 0) continue;
      const BUnit U = decode<KIND>(a, u);
      if (!U.valid || U.ntile == 0) continue;
      for (int t = 0; t < U.ntile; ++t, ++g) {
        const int ks = g % Cfg::kKSlots, vs = g % Cfg::kVSlots;
        if (g >= Cfg::kKSlots && !mbar_wait_nap(&k_empty[ks], (g / Cfg::kKSlots - 1) & 1, abort, a.err)) ok = false;
        if (ok && g >= Cfg::kVSlots && !mbar_wait_nap(&v_empty[vs], (g / Cfg::kVSlots - 1) & 1, abort, a.err))
          ok = false;
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        // key slots (group) or key tokens (window) from key0 + t * 128
        const int y = U.key0 + t * kT;
        if (lane == 0) {
          uint8_t* dk = smem + Cfg::kK + ks * Cfg::kTile;
          uint8_t* dv = smem + Cfg::kV + vs * Cfg::kTile;
          mbar_expect_tx(&k_full[ks], Cfg::kTile);
#pragma unroll
          for (int ch = 0; ch < kChunks; ++ch) tma_load_3d(dk + ch * Cfg::kChunk, &tm_k, &k_full[ks], ch * 64, y, U.zkv);
          mbar_expect_tx(&v_full[vs], Cfg::kTile);
#pragma unroll
          for (int ch = 0; ch < kChunks; ++ch) tma_load_3d(dv + ch * Cfg::kChunk, &tm_v, &v_full[vs], ch * 64, y, U.zkv);
        }
        if (t == 0) {
          // the unit's Q and dO rows, once the previous unit's last S and dP are done
          if (uf > 0 && !mbar_wait_nap(fixed_empty, (uf - 1) & 1, abort, a.err)) ok = false;
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) {
            ++g;
            break;
          }
          if (lane == 0) {
            mbar_expect_tx(fixed_full, 2 * Cfg::kTile);
#pragma unroll
            for (int ch = 0; ch < kChunks; ++ch) {
              tma_load_3d(smem + Cfg::kF0 + ch * Cfg::kChunk, &tm_q, fixed_full, ch * 64, U.row0, U.zq);
              tma_load_3d(smem + Cfg::kF1 + ch * Cfg::kChunk, &tm_do, fixed_full, ch * 64, U.row0, U.zq);
            }
          }
          ++uf;
        }
      }
    }
    if ((*abort || !ok) && lane == 0) {
      // copies already issued must land before the CTA exits
      if (uf > 0) {
        const unsigned long long t0 = global_ns();
        while (!mbar_try_wait(fixed_full, (uf - 1) & 1) && global_ns() - t0 < kWaitTimeoutNs) {}
      }
      for (int x = max(0, g - Cfg::kKSlots); x < g; ++x) {
        const unsigned long long t1 = global_ns();
        while (!mbar_try_wait(&k_full[x % Cfg::kKSlots], (x / Cfg::kKSlots) & 1) && global_ns() - t1 < kWaitTimeoutNs) {}
      }
      for (int x = max(0, g - Cfg::kVSlots); x < g; ++x) {
        const unsigned long long t1 = global_ns();
        while (!mbar_try_wait(&v_full[x % Cfg::kVSlots], (x / Cfg::kVSlots) & 1) && global_ns() - t1 < kWaitTimeoutNs) {}
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------- MMAs ---
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, kT, false, false);
      constexpr uint32_t idAcc = idesc_bf16_f32(128, D, false, true);
      constexpr uint32_t dhi = sw128_desc_hi();
      const uint32_t f0 = sw128_desc_lo(smem_u32(smem + Cfg::kF0), 16);
      const uint32_t f1 = sw128_desc_lo(smem_u32(smem + Cfg::kF1), 16);
      // dQ += dS(x) K(x): the tile's K rows as the MN-major operand
      auto dq_product = [&](int x, bool first, bool last) -> bool {
        if (!mbar_wait_nap(&ew_done[x & 1], (x >> 1) & 1, abort, a.err)) return false;
        tc_fence_after();
        const uint32_t km = sw128_desc_lo(smem_u32(smem + Cfg::kK + (x % Cfg::kKSlots) * Cfg::kTile), Cfg::kChunk);
#pragma unroll
        for (int kk = 0; kk < kT / 16; ++kk)
          mma_ts(tmem + Cfg::kA, tmem + Cfg::kDS + 64 * (x & 1) + kk * 8,
                 desc_join(km + kk * ((16 * 128) >> 4), dhi), idAcc, !first || kk > 0);
        mma_commit(&k_empty[x % Cfg::kKSlots]);
        if (last) mma_commit(acc_full);
        return true;
      };
      bool ok = true;
      int g = 0, uf = 0;
      for (int k = 0; ok; ++k) {
        const int u = bwd_snake(k, n_units);
        if (u == -1) break;
        if (u < 0) continue;
        const BUnit U = decode<KIND>(a, u);
        if (!U.valid || U.ntile == 0) continue;
        if (!mbar_wait_nap(fixed_full, uf & 1, abort, a.err)) { ok = false; break; }
        ++uf;
        for (int t = 0; t < U.ntile; ++t, ++g) {
          const int ks = g % Cfg::kKSlots, vs = g % Cfg::kVSlots;
          if (!mbar_wait_nap(&k_full[ks], (g / Cfg::kKSlots) & 1, abort, a.err) ||
              !mbar_wait_nap(&v_full[vs], (g / Cfg::kVSlots) & 1, abort, a.err) ||
              (g > 0 && !mbar_wait_nap(read_done, (g - 1) & 1, abort, a.err))) {
            ok = false;
            break;
          }
          tc_fence_after();
          // S = Q K^T, dP = dO V^T (both operands K-major over d)
          const uint32_t kb = sw128_desc_lo(smem_u32(smem + Cfg::kK + ks * Cfg::kTile), 16);
          const uint32_t vb = sw128_desc_lo(smem_u32(smem + Cfg::kV + vs * Cfg::kTile), 16);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * Cfg::kChunk + (kk & 3) * 32) >> 4;
            mma_ss(tmem + Cfg::kS, desc_join(f0 + off, dhi), desc_join(kb + off, dhi), idS, kk > 0);
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * Cfg::kChunk + (kk & 3) * 32) >> 4;
            mma_ss(tmem + Cfg::kDP, desc_join(f1 + off, dhi), desc_join(vb + off, dhi), idS, kk > 0);
          }
          mma_commit(sp_full);
          mma_commit(&v_empty[vs]);
          if (t == U.ntile - 1) mma_commit(fixed_empty);
          // the previous tile's product, now that this tile's S and dP are queued
          if (t > 0 && !dq_product(g - 1, t == 1, false)) { ok = false; break; }
        }
        if (!ok) break;
        if (!dq_product(g - 1, U.ntile == 1, true)) { ok = false; break; }
      }
      // every MMA issued above has finished before TMEM is released
      mma_commit(mma_done);
      const unsigned long long t0 = global_ns();
      while (!mbar_try_wait(mma_done, 0) && global_ns() - t0 < kWaitTimeoutNs) {}
    }
  } else if (warp < kEwWarps) {
    // ------------------------------------------------------ elementwise ---
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int r = (warp & 3) * 32 + lane;
    const int half = (warp >> 2) & 1;   // which half of the columns
    const float sl2 = a.scale_log2;
    bool ok = true;
    int g = 0, uf = 0;
    for (int k = 0; ok; ++k) {
      const int u = bwd_snake(k, n_units);
      if (u == -1) break;
      if (u < 0) continue;
      const BUnit U = decode<KIND>(a, u);
      if (!U.valid) continue;
      const size_t pn = static_cast<size_t>(U.prob) * a.n;
      const bool row_ok = r < U.nrows;
      int rpos = -1, klo = 1, khi = 0;
      float lse2 = 0.f, dlt = 0.f;
      if (row_ok) {
        if (KIND == kDqGroup) {
          rpos = a.perm[pn + U.row0 + r];
          klo = 0;
          khi = a.farlen_slot[pn + U.row0 + r] - 1;       // prefix index
        } else {
          rpos = U.row0 + r;
          klo = rpos - a.w + 1;
          khi = rpos;                                     // key tokens
        }
        const size_t qi = static_cast<size_t>(U.zq) * a.n + rpos;
        lse2 = a.lse[qi] * kLog2e;
        dlt = a.delta[qi];
      }
      for (int t = 0; t < U.ntile; ++t, ++g) {
        if (!warp_wait(sp_full, g & 1, abort, a.err)) { ok = false; break; }
        tc_fence_after();
        // this half's 64 columns of S and dP
        uint32_t sv[64], dv[64];
        tmem_ld32(tmem + lane_base + Cfg::kS + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
        tmem_ld32(tmem + lane_base + Cfg::kS + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
        tmem_ld32(tmem + lane_base + Cfg::kDP + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&dv[0]));
        tmem_ld32(tmem + lane_base + Cfg::kDP + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&dv[32]));
        tmem_wait_ld();
        tc_fence_before();
        warp_arrive(read_done, lane);
        uint32_t dd[32];
        const int base_idx = (KIND == kDqGroup ? 0 : U.key0) + t * kT + half * 64;
#pragma unroll
        for (int e = 0; e < 64; e += 2) {
          float d2[2];
#pragma unroll
          for (int q2 = 0; q2 < 2; ++q2) {
            const int idx = base_idx + e + q2;
            const bool keep = row_ok && idx >= klo && idx <= khi;
            const float p = keep ? ex2f(__uint_as_float(sv[e + q2]) * sl2 - lse2) : 0.f;
            d2[q2] = p * (__uint_as_float(dv[e + q2]) - dlt);
          }
          dd[e / 2] = pack_bf16x2(d2[0], d2[1]);
        }
        // the half's 64 bf16 values take packed columns 32*half .. 32*half + 31 of dS(g)
        tmem_st32(tmem + lane_base + Cfg::kDS + 64 * (g & 1) + half * 32, dd);
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(&ew_done[g & 1], lane);
      }
      if (!ok) break;
      // epilogue: this half's dQ columns [half * D/2, (half + 1) * D/2) once the unit's products are done
      const bool have = U.ntile > 0;
      if (have) {
        if (!warp_wait(acc_full, uf & 1, abort, a.err)) { ok = false; break; }
        ++uf;
        tc_fence_after();
      }
      const size_t orow = static_cast<size_t>(U.zq) * a.n + (rpos >= 0 ? rpos : 0);
#pragma unroll 1
      for (int c = half * (D / 64); c < (half + 1) * (D / 64); ++c) {
        uint32_t x0[32];
        if (have) {
          tmem_ld32(tmem + lane_base + Cfg::kA + c * 32, x0);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) x0[e] = 0u;
        }
        if (!row_ok) continue;
        const size_t o = orow * D + c * 32;
        if (KIND == kDqGroup) {
          float4* dst = reinterpret_cast<float4*>(a.dq_far + o);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            dst[v] = make_float4(__uint_as_float(x0[4 * v]) * a.scale, __uint_as_float(x0[4 * v + 1]) * a.scale,
                                 __uint_as_float(x0[4 * v + 2]) * a.scale, __uint_as_float(x0[4 * v + 3]) * a.scale);
        } else {
          const bool far = a.farlen_tok[pn + rpos] > 0;
          const float4* fq = reinterpret_cast<const float4*>(a.dq_far + o);
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.dQ) + o);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            float f[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(x0[8 * v + e]) * a.scale;
            if (far) {
              const float4 g0 = fq[2 * v], g1 = fq[2 * v + 1];
              f[0] += g0.x; f[1] += g0.y; f[2] += g0.z; f[3] += g0.w;
              f[4] += g1.x; f[5] += g1.y; f[6] += g1.z; f[7] += g1.w;
            }
            dst[v] = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                                pack_bf16x2(f[6], f[7]));
          }
        }
      }
      tc_fence_before();
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Q, dO rows and the LSE, Delta of every query head in the order of its
// assignment's index: dst[zq, s] = src[zq, perm_a[s]], a = the head's assignment.
__global__ void __launch_bounds__(256) permute_q_kernel(BwdArgs a, __nv_bfloat16* Qs, __nv_bfloat16* dOs,
                                                        float* lse_s, float* delta_s, long long total) {
  const int vpr = a.d / 8;
  for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = e / vpr;
    const int u = static_cast<int>(e % vpr);
    const int s = static_cast<int>(row % a.n);
    const long long zq = row / a.n;
    const int h = static_cast<int>(zq % a.H);
    const long long b = zq / a.H;
    const long long p = b * a.A + (a.A == 1 ? 0 : (h * a.H_kv) / a.H);
    const long long src = zq * a.n + __ldg(a.perm + p * a.n + s);
    reinterpret_cast<uint4*>(Qs)[e] = __ldg(reinterpret_cast<const uint4*>(a.Q) + src * vpr + u);
    reinterpret_cast<uint4*>(dOs)[e] = __ldg(reinterpret_cast<const uint4*>(a.dO) + src * vpr + u);
    if (u == 0) {
      lse_s[row] = a.lse[src];
      delta_s[row] = a.delta[src];
    }
  }
}

template <int D>
cudaError_t launch_d(const BwdArgs& a, const CUtensorMap* qs, const CUtensorMap* dos, const CUtensorMap* ks,
                     const CUtensorMap* vs, const CUtensorMap* q3, const CUtensorMap* do3, const CUtensorMap* k3,
                     const CUtensorMap* v3, int max_items, int num_sms, cudaStream_t st) {
  using Cfg = BCfg<D>;
  const int hpa = a.A == 1 ? a.H : a.H / a.H_kv;
  const long long g_units = static_cast<long long>(max_items) * hpa;
  const long long q_units = static_cast<long long>(a.B) * a.H * ((a.n + kT - 1) / kT);
  const long long k_units = static_cast<long long>(a.B) * a.H_kv * ((a.n + kT - 1) / kT);
  const long long sms = num_sms > 0 ? num_sms : 1;
  if (g_units > 0)
    bwd_dq_kernel<D, kDqGroup><<<static_cast<unsigned>(std::min(g_units, sms)), kThreads, DqCfg<D>::kSmem, st>>>(
        *qs, *dos, *ks, *vs, a);
  bwd_dq_kernel<D, kDqLocal><<<static_cast<unsigned>(std::min(q_units, sms)), kThreads, DqCfg<D>::kSmem, st>>>(
      *q3, *do3, *k3, *v3, a);
  bwd_tc_kernel<D, kDkvGroup><<<static_cast<unsigned>(k_units), kThreads, Cfg::kSmem, st>>>(*qs, *dos, *ks, *vs, a);
  bwd_tc_kernel<D, kDkvLocal><<<static_cast<unsigned>(k_units), kThreads, Cfg::kSmem, st>>>(*q3, *do3, *k3, *v3, a);
  return cudaGetLastError();
}

template <int D>
cudaError_t set_smem_d() {
  using Cfg = BCfg<D>;
  cudaError_t e;
  e = cudaFuncSetAttribute(bwd_dq_kernel<D, kDqGroup>, cudaFuncAttributeMaxDynamicSharedMemorySize, DqCfg<D>::kSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(bwd_dq_kernel<D, kDqLocal>, cudaFuncAttributeMaxDynamicSharedMemorySize, DqCfg<D>::kSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(bwd_tc_kernel<D, kDkvGroup>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(bwd_tc_kernel<D, kDkvLocal>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
}

}  // namespace

cudaError_t launch_attn_bwd_tc(const BwdArgs& a, const CUtensorMap* qs, const CUtensorMap* dos,
                               const CUtensorMap* ks, const CUtensorMap* vs, const CUtensorMap* q3,
                               const CUtensorMap* do3, const CUtensorMap* k3, const CUtensorMap* v3,
                               int max_items, int num_sms, cudaStream_t st) {
  if (a.d == 64) return launch_d<64>(a, qs, dos, ks, vs, q3, do3, k3, v3, max_items, num_sms, st);
  if (a.d == 128) return launch_d<128>(a, qs, dos, ks, vs, q3, do3, k3, v3, max_items, num_sms, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_permute_q(const BwdArgs& a, void* Qs, void* dOs, float* lse_s, float* delta_s,
                                 cudaStream_t st) {
  const long long total = static_cast<long long>(a.B) * a.H * a.n * (a.d / 8);
  const long long want = (total + 255) / 256;
  const int grid = static_cast<int>(want < 152LL * 16 ? want : 152LL * 16);
  permute_q_kernel<<<grid, 256, 0, st>>>(a, static_cast<__nv_bfloat16*>(Qs), static_cast<__nv_bfloat16*>(dOs),
                                         lse_s, delta_s, total);
  return cudaGetLastError();
}

cudaError_t setup_bwd_tc_kernels() {
  cudaError_t e = set_smem_d<64>();
  if (e != cudaSuccess) return e;
  return set_smem_d<128>();
}

}  // namespace focus
