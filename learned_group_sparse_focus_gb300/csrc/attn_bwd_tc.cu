// Backward of Focus attention on the tcgen05 tensor cores (bf16 tensors, fp32
// accumulate): the same gradients as attn_bwd.cu ("Why Attend to Everything?
// Focus is the Key", section 2.1; "Focus: Learning Which Attention Pairs
// Matter", section 3.1), with every d-long product an MMA.
//
// Two persistent kernels (one CTA per SM looping over 128-row units), each in
// a group form (far pairs, rows and keys in the index's sorted order, read as
// TMA tiles from copies of Q, dO, K, V (and LSE, Delta) sorted by the index
// once per call) and a window form (natural order, TMA tiles):
//   dQ   rows = 128 queries, streamed = 128-key tiles of the kept keys:
//          S = Q K^T, dP = dO V^T               (SS, TMEM fp32)
//          dS = P (dP - Delta), P = exp(S scale - LSE)   (CUDA cores -> TMEM bf16)
//          dQ += dS K                           (TS, K as the MN-major operand)
//   dKV  rows = 128 keys, streamed = 128-query tiles of the queries that keep
//        them, for every query head of the key/value head:
//          S^T = K Q^T, dP^T = V dO^T           (SS)
//          P^T, dS^T                            (CUDA cores -> TMEM bf16)
//          dV += P^T dO, dK += dS^T Q           (TS)
// Warps 0-7 do the elementwise work, two per TMEM lane quadrant, each on half
// of the row's columns; warp 8 loads, warp 9 owns TMEM and issues the MMAs.
// Each kernel keeps the tensor pipe busy while the elementwise warps work (its
// own comment says how).  Every wait is bounded; on a timeout the CTA raises
// the error bit, drains its copies, frees TMEM and exits.
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

__device__ __forceinline__ void prefetch_l2(const float* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

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

// dQ far unit u (item order[u / hpa], query head u % hpa of its assignment) from its item.
__device__ __forceinline__ BUnit decode_item(const BwdArgs& a, int u, const focus_item_t& it) {
  BUnit U{};
  U.valid = true;
  U.heads = 1;
  const int hpa = a.A == 1 ? a.H : a.H / a.H_kv;
  const int y = u % hpa;
  U.b = it.b;
  U.h = a.A == 1 ? y : it.a * (a.H / a.H_kv) + y;
  U.kv = (U.h * a.H_kv) / a.H;
  U.prob = it.b * a.A + it.a;
  U.row0 = it.row0;
  U.nrows = it.rows;
  U.key0 = it.key0;
  U.nkeys = it.keys;
  U.ntile = (it.keys + kT - 1) / kT;
  U.zq = U.b * a.H + U.h;
  U.zkv = U.b * a.H_kv + U.kv;
  return U;
}

template <int KIND>
__device__ __forceinline__ BUnit decode(const BwdArgs& a, int u) {
  BUnit U{};
  U.valid = true;
  U.heads = 1;
  if (KIND == kDqGroup) {
    const int io = u / (a.A == 1 ? a.H : a.H / a.H_kv);
    if (io >= *a.n_items) {
      U.valid = false;
      return U;
    }
    return decode_item(a, u, a.items[a.order[io]]);
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
  uint64_t* stage_free = bars + 18;   // [2] by unit parity: the unit's epilogue is done with its slabs
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
    mbar_init(&stage_free[0], kEwWarps);
    mbar_init(&stage_free[1], kEwWarps);
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
    // A unit's epilogue stages its rows in the V slot of the unit's last tile
    // L; the V load of tile L + 2, the next into that slot, waits for it.
    // Pending targets L + 2, oldest first (at most two: every unit has a tile).
    // The barrier alternates with the unit: the epilogue two units later needs
    // the V load of a tile past L + 2, so neither runs a phase ahead.
    int st0 = -1, st1 = -1, sw = 0;
    int kv_half = 0;   // set when the loop stops with tile g's V issued and its K not
    for (int k = 0; ok; ++k) {
      const int u = bwd_snake(k, n_units);
      if (u == -1) break;
      if (u < 0) continue;
      const BUnit U = decode<KIND>(a, u);
      if (!U.valid || U.ntile == 0) continue;
      for (int t = 0; t < U.ntile; ++t, ++g) {
        const int ks = g % Cfg::kKSlots, vs = g % Cfg::kVSlots;
        // key slots (group) or key tokens (window) from key0 + t * 128; V first:
        // its slot frees when the S and dP products are done, K's only after
        // the dQ product
        const int y = U.key0 + t * kT;
        if (g >= Cfg::kVSlots && !mbar_wait_nap(&v_empty[vs], (g / Cfg::kVSlots - 1) & 1, abort, a.err)) ok = false;
        if (ok && g == st0) {
          if (!mbar_wait_nap(&stage_free[sw & 1], (sw >> 1) & 1, abort, a.err)) ok = false;
          ++sw;
          st0 = st1;
          st1 = -1;
        }
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        if (lane == 0) {
          uint8_t* dv = smem + Cfg::kV + vs * Cfg::kTile;
          mbar_expect_tx(&v_full[vs], Cfg::kTile);
#pragma unroll
          for (int ch = 0; ch < kChunks; ++ch) tma_load_3d(dv + ch * Cfg::kChunk, &tm_v, &v_full[vs], ch * 64, y, U.zkv);
        }
        if (g >= Cfg::kKSlots && !mbar_wait_nap(&k_empty[ks], (g / Cfg::kKSlots - 1) & 1, abort, a.err)) ok = false;
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
          kv_half = 1;   // V of tile g is in flight, K is not
          break;
        }
        if (lane == 0) {
          uint8_t* dk = smem + Cfg::kK + ks * Cfg::kTile;
          mbar_expect_tx(&k_full[ks], Cfg::kTile);
#pragma unroll
          for (int ch = 0; ch < kChunks; ++ch) tma_load_3d(dk + ch * Cfg::kChunk, &tm_k, &k_full[ks], ch * 64, y, U.zkv);
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
      if (!ok) break;
      if (st0 < 0) st0 = g + 1; else st1 = g + 1;   // this unit's L + 2 (g = L + 1 here)
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
      for (int x = max(0, g + kv_half - Cfg::kVSlots); x < g + kv_half; ++x) {
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
    // window kind: the next unit's LSE, Delta and far flag, loaded one unit ahead
    int nu = -1;
    float n_lse = 0.f, n_dlt = 0.f;
    bool n_far = false;
    // group kind: the next unit is named by a chain of dependent loads (order
    // entry, item, then the row's slot and far length, then its LSE and
    // Delta); one link is issued per tile of this unit, so the chain is done
    // by the time the next unit starts
    int gq_u = -1, gq_stage = 0, gq_ord = 0, gq_rpos = -1, gq_khi = 0;
    focus_item_t gq_it{};
    BUnit GU{};
    float gq_lse = 0.f, gq_dlt = 0.f;
    auto gq_advance = [&]() {
      if (gq_stage == 1) {
        gq_it = a.items[gq_ord];
      } else if (gq_stage == 2) {
        GU = decode_item(a, gq_u, gq_it);
        if (r < GU.nrows) {
          const size_t at = static_cast<size_t>(GU.prob) * a.n + GU.row0 + r;
          gq_rpos = a.perm[at];
          gq_khi = a.farlen_slot[at] - 1;
        }
      } else if (gq_stage == 3 && r < GU.nrows) {
        const size_t qi = static_cast<size_t>(GU.zq) * a.n + gq_rpos;
        gq_lse = a.lse[qi];
        gq_dlt = a.delta[qi];
      }
      ++gq_stage;
    };
    for (int k = 0; ok; ++k) {
      const int u = bwd_snake(k, n_units);
      if (u == -1) break;
      if (u < 0) continue;
      const bool pre = KIND == kDqGroup && u == gq_u && gq_stage == 4;
      const BUnit U = pre ? GU : decode<KIND>(a, u);
      if (!U.valid) continue;
      const size_t pn = static_cast<size_t>(U.prob) * a.n;
      const bool row_ok = r < U.nrows;
      int rpos = -1, klo = 1, khi = 0;
      float lse2 = 0.f, dlt = 0.f;
      bool far = false;
      if (pre) {
        if (row_ok) {
          rpos = gq_rpos;
          klo = 0;
          khi = gq_khi;
          lse2 = gq_lse * kLog2e;
          dlt = gq_dlt;
        }
      } else if (KIND == kDqLocal && u == nu) {
        if (row_ok) {
          rpos = U.row0 + r;
          klo = rpos - a.w + 1;
          khi = rpos;
          lse2 = n_lse * kLog2e;
          dlt = n_dlt;
          far = n_far;
        }
      } else if (row_ok) {
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
        if (KIND == kDqLocal) far = a.farlen_tok[pn + rpos] > 0;   // read by the epilogue
      }
      if (KIND == kDqGroup) {
        // start the next unit's chain: its order entry now
        gq_u = bwd_snake(k + 1, n_units);
        gq_stage = 0;
        if (gq_u >= 0) {
          gq_ord = a.order[gq_u / (a.A == 1 ? a.H : a.H / a.H_kv)];
          gq_stage = 1;
        }
      }
      if (KIND == kDqLocal) {
        nu = bwd_snake(k + 1, n_units);
        if (nu >= 0) {
          const BUnit N = decode<KIND>(a, nu);
          if (r < N.nrows) {
            const size_t qi = static_cast<size_t>(N.zq) * a.n + N.row0 + r;
            n_lse = a.lse[qi];
            n_dlt = a.delta[qi];
            n_far = a.farlen_tok[static_cast<size_t>(N.prob) * a.n + N.row0 + r] > 0;
          }
        }
      }
      const uint64_t sc2 = f2_pack(sl2, sl2), nl2 = f2_pack(-lse2, -lse2), nd2 = f2_pack(-dlt, -dlt);
      for (int t = 0; t < U.ntile; ++t, ++g) {
        if (KIND == kDqLocal && far && t == max(0, U.ntile - 3)) {
          // the epilogue's far part, three tiles ahead so that it is in L2 when read
          const size_t o = (static_cast<size_t>(U.zq) * a.n + rpos) * D + half * (D / 2);
#pragma unroll
          for (int q = 0; q < D / 2; q += 32) prefetch_l2(a.dq_far + o + q);
        }
        const int c0 = (KIND == kDqGroup ? 0 : U.key0) + t * kT + half * 64;   // key index of column 0
        // bit e: the row keeps column c0 + e
        const int lo = max(klo - c0, 0), hi = min(khi - c0, 63);
        const uint64_t keepm = (row_ok && lo <= hi) ? ((~0ull >> (63 - hi)) & (~0ull << lo)) : 0ull;
        const bool full = __all_sync(0xffffffffu, keepm == ~0ull);
        if (!warp_wait(sp_full, g & 1, abort, a.err)) { ok = false; break; }
        tc_fence_after();
        // this half's 64 columns of S and dP, 32 at a time (the second pair of
        // reads releases S and dP to the next tile's products); dS = P (dP - Delta)
        // with P = 2^(s scale log2e - lse2) in packed pairs, a dropped pair
        // getting exp2(-inf) = +0 with no branch around the exponential
        uint32_t dd[32];
#pragma unroll
        for (int hq = 0; hq < 2; ++hq) {
          uint32_t sv[32], dv[32];
          tmem_ld32(tmem + lane_base + Cfg::kS + half * 64 + 32 * hq, sv);
          tmem_ld32(tmem + lane_base + Cfg::kDP + half * 64 + 32 * hq, dv);
          tmem_wait_ld();
          if (hq == 1) {
            tc_fence_before();
            warp_arrive(read_done, lane);
          }
          if (full) {
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              float t0, t1, d0, d1;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), sc2, nl2), t0, t1);
              const uint64_t q = f2_pack(ex2f(t0), ex2f(t1));
              f2_unpack(f2_mul(q, f2_add(f2_pack(__uint_as_float(dv[e]), __uint_as_float(dv[e + 1])), nd2)), d0, d1);
              dd[16 * hq + e / 2] = pack_bf16x2(d0, d1);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const int b0 = 32 * hq + e;
              float t0, t1, d0, d1;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), sc2, nl2), t0, t1);
              const uint64_t q = f2_pack(ex2f((keepm >> b0) & 1 ? t0 : -INFINITY),
                                         ex2f((keepm >> (b0 + 1)) & 1 ? t1 : -INFINITY));
              f2_unpack(f2_mul(q, f2_add(f2_pack(__uint_as_float(dv[e]), __uint_as_float(dv[e + 1])), nd2)), d0, d1);
              dd[16 * hq + e / 2] = pack_bf16x2(d0, d1);
            }
          }
        }
        // the half's 64 bf16 values take packed columns 32*half .. 32*half + 31 of dS(g)
        tmem_st32(tmem + lane_base + Cfg::kDS + 64 * (g & 1) + half * 32, dd);
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(&ew_done[g & 1], lane);
        if (KIND == kDqGroup && gq_stage > 0 && gq_stage < 4) gq_advance();
      }
      if (!ok) break;
      // Epilogue: this half's dQ columns [half * D/2, (half + 1) * D/2) once the
      // unit's products are done.  A unit with no tiles (group kind) has no
      // far keys in any row, and the window kernel reads none of its rows.
      // one more link of the next unit's chain, its latency under the epilogue
      if (KIND == kDqGroup && gq_stage > 0 && gq_stage < 4) gq_advance();
      if (U.ntile == 0) continue;
      if (!warp_wait(acc_full, uf & 1, abort, a.err)) { ok = false; break; }
      ++uf;
      tc_fence_after();
      // Each thread holds its row's values; they go through this warp's 32 x 16
      // fp32 slab (16-byte pieces at slot piece ^ ((row >> 1) & 3), so neither
      // the row writes nor the column reads conflict) in the V slot of the
      // unit's last tile, which its products no longer read and the loader
      // refills only after stage_free, and leave as 64-byte runs of one row per
      // four lanes.
      float* stg = reinterpret_cast<float*>(smem + Cfg::kV + ((g - 1) % Cfg::kVSlots) * Cfg::kTile) + warp * 512;
      const int jr = lane >> 2, kq = lane & 3;
      const size_t zrow = static_cast<size_t>(U.zq) * a.n;
      int rp4[4];          // token of pass row 8i + jr
      bool ok4[4], far4[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        rp4[i] = __shfl_sync(0xffffffffu, rpos, 8 * i + jr);
        far4[i] = __shfl_sync(0xffffffffu, far ? 1 : 0, 8 * i + jr) != 0;
        ok4[i] = (warp & 3) * 32 + 8 * i + jr < U.nrows;
      }
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {      // this half's 32-column groups
        const int c = half * (D / 64) + cc;
        // window kind: the far part of the group's eight row pieces, in flight
        // while the accumulator is read and staged
        float4 fv[8];
        if (KIND == kDqLocal) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int i = q & 3, s16 = q >> 2;
            fv[q] = ok4[i] && far4[i]
                        ? *reinterpret_cast<const float4*>(a.dq_far + (zrow + rp4[i]) * D + c * 32 + s16 * 16 + 4 * kq)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
        uint32_t x[32];
        tmem_ld32(tmem + lane_base + Cfg::kA + c * 32, x);
        tmem_wait_ld();
#pragma unroll
        for (int s16 = 0; s16 < 2; ++s16) {      // 16-column pieces of the 32
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int e = 16 * s16 + 4 * k;
            *reinterpret_cast<float4*>(stg + lane * 16 + 4 * (k ^ ((lane >> 1) & 3))) =
                make_float4(__uint_as_float(x[e]) * a.scale, __uint_as_float(x[e + 1]) * a.scale,
                            __uint_as_float(x[e + 2]) * a.scale, __uint_as_float(x[e + 3]) * a.scale);
          }
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int j = 8 * i + jr;              // row of this warp's 32
            const float4 v = *reinterpret_cast<const float4*>(stg + j * 16 + 4 * (kq ^ ((j >> 1) & 3)));
            if (ok4[i]) {
              const size_t o = (zrow + rp4[i]) * D + c * 32 + s16 * 16 + 4 * kq;
              if (KIND == kDqGroup) {
                *reinterpret_cast<float4*>(a.dq_far + o) = v;
              } else {
                const float4 f = fv[4 * s16 + i];
                *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.dQ) + o) =
                    make_uint2(pack_bf16x2(v.x + f.x, v.y + f.y), pack_bf16x2(v.z + f.z, v.w + f.w));
              }
            }
          }
        }
      }
      // the slab's generic accesses before the loader's next copy into the slot
      fence_proxy_async_smem();
      warp_arrive(&stage_free[(uf - 1) & 1], lane);
      tc_fence_before();
      // a short unit leaves links of the chain for here
      while (KIND == kDqGroup && gq_stage > 0 && gq_stage < 4) gq_advance();
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
// dK/dV kernels, persistent: one CTA per SM takes units (128 key rows of one
// KV head) from a ticket counter in the longest-first order kv_order_kernel
// writes (group kind) or in snake order (window kind) and walks, for every
// query head of the KV head, the query tiles that keep the unit's keys.  The loader warp names each unit, finds its rows'
// kept query ranges and publishes them through a 2-entry ring in shared
// memory, so the elementwise warps never search at a unit boundary.  TMEM is
// S^T | dP^T | dV | dK; per tile the tensor pipe runs
//   S^T = K Q^T,  dP^T = V dO^T,  dV += P^T dO,  dK += dS^T Q
// and the elementwise warps work in two steps, P^T (over S^T, in place) as
// soon as S^T is there and dS^T (over dP^T) once dP^T is.  The next tile's
// S^T is issued as soon as dV has read P^T, ahead of dK, so it runs while
// dS^T is computed.
template <int D>
struct KvCfg {
  static constexpr int kChunk = 128 * 128;
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kF0 = 0;              // K rows of the unit
  static constexpr int kF1 = kTile;          // V rows of the unit
  static constexpr int kR = 2 * kTile;       // ring: 2 slots x (Q, dO)
  static constexpr int kCol = kR + 4 * kTile;          // [4 slots][-lse2, -delta][128] fp32
  static constexpr int kRow = kCol + 4 * 2 * 128 * 4;  // [2 units][128] (klo, khi)
  static constexpr int kInfo = kRow + 2 * 128 * 8;     // [2 units] {unit, wlo, ntile, -}
  static constexpr int kStage = kInfo + 64;            // [8 warps][32 rows][16] fp32 epilogue slabs
  static constexpr int kBar = kStage + kEwWarps * 32 * 16 * 4;
  static constexpr int kMisc = kBar + 256;
  static constexpr int kBytes = kMisc + 64;
  static constexpr int kSmem = kBytes + 1024;
  static constexpr uint32_t kS = 0, kDP = 128, kDV = 256, kDK = 256 + D;
};
static_assert(KvCfg<128>::kSmem <= 227 * 1024, "dK/dV shared memory above 227 KB");

template <int D, int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                   const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const BwdArgs a) {
  using Cfg = KvCfg<D>;
  constexpr int kChunks = D / 64;
  constexpr bool kGroup = KIND == kDkvGroup;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kBar);
  uint64_t* fixed_full = bars + 0;
  uint64_t* fixed_empty = bars + 1;
  uint64_t* ring_full = bars + 2;     // [2]
  uint64_t* ring_empty = bars + 4;    // [2]
  uint64_t* col_full = bars + 6;      // [4] the tile's query LSE / Delta are in shared memory
  uint64_t* s_full = bars + 10;
  uint64_t* dp_full = bars + 11;
  uint64_t* p_done = bars + 12;       // P^T of the tile is in TMEM
  uint64_t* ds_done = bars + 13;      // dS^T of the tile is in TMEM
  uint64_t* v_done = bars + 14;       // dV += P^T dO of the tile is done (S^T columns free)
  uint64_t* k_done = bars + 15;       // dK += dS^T Q of the tile is done (dP^T columns free)
  uint64_t* acc_full = bars + 16;     // the unit's dK, dV are complete
  uint64_t* info_full = bars + 17;    // [2]
  uint64_t* info_empty = bars + 19;   // [2]
  uint64_t* mma_done = bars + 21;
  int* misc = reinterpret_cast<int*>(smem + Cfg::kMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 0);
  volatile int* abort = misc + 1;
  float* colbuf = reinterpret_cast<float*>(smem + Cfg::kCol);
  int2* rowinfo = reinterpret_cast<int2*>(smem + Cfg::kRow);
  int4* info = reinterpret_cast<int4*>(smem + Cfg::kInfo);
  float* stage = reinterpret_cast<float*>(smem + Cfg::kStage);

  const int warp = warp_id(), lane = lane_id();
  const int nkt = (a.n + kT - 1) / kT;
  const int n_units = a.B * a.H_kv * nkt;
  const int heads = a.H / a.H_kv;

  if (threadIdx.x == 0) {
    mbar_init(fixed_full, 1);
    mbar_init(fixed_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&ring_full[s], 1);
      mbar_init(&ring_empty[s], 1);
      mbar_init(&info_full[s], 1);
      mbar_init(&info_empty[s], kEwWarps + 1);
    }
    for (int s = 0; s < 4; ++s) mbar_init(&col_full[s], 32);
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(p_done, kEwWarps);
    mbar_init(ds_done, kEwWarps);
    mbar_init(v_done, 1);
    mbar_init(k_done, 1);
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
    // ------------------------------------------- unit names, ranges, loads ---
    bool ok = true;
    int g = 0, uf = 0, snake = 0;
    // Names unit k, finds every row's kept query range [klo, khi] (slots in the
    // group kind, tokens in the window kind) and publishes both; runs one unit
    // ahead of the loads, so the searches overlap the previous unit's tiles.
    auto name_unit = [&](int k, int& u, BUnit& U, int& wlo, int& ntile) -> bool {
      u = -1;
      if (kGroup) {
        if (lane == 0) {
          const int tk = atomicAdd(a.ticket, 1);
          u = tk < n_units ? a.kv_order[tk] : -1;
        }
        u = __shfl_sync(0xffffffffu, u, 0);
      } else {
        for (;;) {
          u = bwd_snake(snake++, n_units);
          if (u != -2) break;
        }
      }
      bool fine = !(k >= 2 && !mbar_wait_nap(&info_empty[k & 1], ((k >> 1) - 1) & 1, abort, a.err));
      if (!__all_sync(0xffffffffu, fine)) return false;
      wlo = 0;
      ntile = 0;
      int lo = 0x7fffffff, hi = -1;
      if (u >= 0) {
        U = decode<KIND>(a, u);
        const size_t pn = static_cast<size_t>(U.prob) * a.n;
        int klo[4], khi[4];
        if (kGroup) {
          // four rows per lane, their binary searches interleaved
          const int32_t* off = a.offsets + static_cast<size_t>(U.prob) * (a.groups + 1);
          int us[4], tg[4], gl[4], gh[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int rr = lane + 32 * j;
            us[j] = U.row0 + rr;
            const bool v = rr < U.nrows;
            tg[j] = v ? a.perm[pn + us[j]] + a.w : 0;
            gl[j] = 0;
            gh[j] = v ? a.groups : 1;
          }
          for (;;) {   // the slot's group: off[gl] <= slot < off[gl + 1]
            bool more = false;
            int val[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) val[j] = gh[j] - gl[j] > 1 ? off[(gl[j] + gh[j]) >> 1] : 0;
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (gh[j] - gl[j] > 1) {
                const int mid = (gl[j] + gh[j]) >> 1;
                if (val[j] <= us[j]) gl[j] = mid; else gh[j] = mid;
                more = more || gh[j] - gl[j] > 1;
              }
            if (!more) break;
          }
          int s0[4], s1[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const bool v = lane + 32 * j < U.nrows;
            s1[j] = v ? off[gl[j] + 1] : 0;
            s0[j] = v ? us[j] + 1 : 0;
            khi[j] = v ? s1[j] - 1 : 0;
            if (!v) {
              s0[j] = 1;
              s1[j] = 1;
            }
          }
          for (;;) {   // first later slot of the group at or past position + w
            bool more = false;
            int val[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) val[j] = s0[j] < s1[j] ? a.perm[pn + ((s0[j] + s1[j]) >> 1)] : 0;
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (s0[j] < s1[j]) {
                const int mid = (s0[j] + s1[j]) >> 1;
                if (val[j] < tg[j]) s0[j] = mid + 1; else s1[j] = mid;
                more = more || s0[j] < s1[j];
              }
            if (!more) break;
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) klo[j] = s0[j];
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int rp = U.row0 + lane + 32 * j;
            klo[j] = rp;
            khi[j] = min(a.n - 1, rp + a.w - 1);
          }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int rr = lane + 32 * j;
          if (rr >= U.nrows) {
            klo[j] = 1;
            khi[j] = 0;
          }
          rowinfo[(k & 1) * 128 + rr] = make_int2(klo[j], khi[j]);
          if (klo[j] <= khi[j]) {
            lo = min(lo, klo[j]);
            hi = max(hi, khi[j]);
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
          hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
        }
        if (hi >= lo) {
          wlo = lo;
          ntile = (hi - lo) / kT + 1;
        }
      }
      if (lane == 0) info[k & 1] = make_int4(u, wlo, ntile, 0);
      __syncwarp();
      if (lane == 0) mbar_arrive(&info_full[k & 1]);
      return true;
    };
    int u = -1, wlo = 0, ntile = 0;
    BUnit U{};
    ok = name_unit(0, u, U, wlo, ntile);
    for (int k = 0; ok && u >= 0; ++k) {
      int u1 = -1, wlo1 = 0, ntile1 = 0;
      BUnit U1{};
      if (!name_unit(k + 1, u1, U1, wlo1, ntile1)) {
        ok = false;
        break;
      }
      const int ntot = ntile * heads;
      for (int i = 0, t = 0, hh = 0; i < ntot; ++i, ++g) {
        const int sl = g & 1;
        const int zq = U.b * a.H + U.h + hh;
        const int y = wlo + t * kT;
        // the tile's query columns: -LSE (log2 units) and -Delta of head h + hh,
        // read from global memory before the ring wait and stored after it
        float l2[4], dl[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int q = y + 4 * lane + j;
          l2[j] = dl[j] = 0.f;
          if (q < a.n) {
            const size_t qi = static_cast<size_t>(zq) * a.n + q;
            l2[j] = (kGroup ? a.lse_sorted : a.lse)[qi];
            dl[j] = (kGroup ? a.delta_sorted : a.delta)[qi];
          }
        }
        if (g >= 2 && !mbar_wait_nap(&ring_empty[sl], ((g >> 1) - 1) & 1, abort, a.err)) ok = false;
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        uint8_t* r0 = smem + Cfg::kR + sl * 2 * Cfg::kTile;
        if (lane == 0) {
          mbar_expect_tx(&ring_full[sl], 2 * Cfg::kTile);
#pragma unroll
          for (int ch = 0; ch < kChunks; ++ch) {
            tma_load_3d(r0 + ch * Cfg::kChunk, &tm_q, &ring_full[sl], ch * 64, y, zq);
            tma_load_3d(r0 + Cfg::kTile + ch * Cfg::kChunk, &tm_do, &ring_full[sl], ch * 64, y, zq);
          }
        }
        float* cb = colbuf + (g & 3) * 256;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          cb[4 * lane + j] = -l2[j] * kLog2e;
          cb[128 + 4 * lane + j] = -dl[j];
        }
        mbar_arrive(&col_full[g & 3]);
        if (++t == ntile) {
          t = 0;
          ++hh;
        }
        if (i == 0) {
          // the unit's K and V rows, once the previous unit's last S^T and dP^T are done
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
              tma_load_3d(smem + Cfg::kF0 + ch * Cfg::kChunk, &tm_k, fixed_full, ch * 64, U.row0, U.zkv);
              tma_load_3d(smem + Cfg::kF1 + ch * Cfg::kChunk, &tm_v, fixed_full, ch * 64, U.row0, U.zkv);
            }
          }
          ++uf;
        }
      }
      u = u1;
      U = U1;
      wlo = wlo1;
      ntile = ntile1;
    }
    if ((*abort || !ok) && lane == 0) {
      // copies already issued must land before the CTA exits
      if (uf > 0) {
        const unsigned long long t0 = global_ns();
        while (!mbar_try_wait(fixed_full, (uf - 1) & 1) && global_ns() - t0 < kWaitTimeoutNs) {}
      }
      for (int x = max(0, g - 2); x < g; ++x) {
        const unsigned long long t1 = global_ns();
        while (!mbar_try_wait(&ring_full[x & 1], (x >> 1) & 1) && global_ns() - t1 < kWaitTimeoutNs) {}
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------- MMAs ---
    bool ok = true;
    int g = 0, uf = 0;
    constexpr uint32_t idS = idesc_bf16_f32(128, kT, false, false);
    constexpr uint32_t idAcc = idesc_bf16_f32(128, D, false, true);
    constexpr uint32_t dhi = sw128_desc_hi();
    const uint32_t f0 = sw128_desc_lo(smem_u32(smem + Cfg::kF0), 16);
    const uint32_t f1 = sw128_desc_lo(smem_u32(smem + Cfg::kF1), 16);
    for (int k = 0; ok; ++k) {
      if (!warp_wait(&info_full[k & 1], (k >> 1) & 1, abort, a.err)) { ok = false; break; }
      const int4 in = info[k & 1];
      warp_arrive(&info_empty[k & 1], lane);
      if (in.x < 0) break;
      const int ntot = in.z * heads;
      if (ntot == 0) continue;
      if (lane == 0) {
        // S^T = K Q^T of tile x into TMEM columns 0..127, once dV of tile x - 1 has read its P^T
        auto issue_s = [&](int x) -> bool {
          if (!mbar_wait_nap(&ring_full[x & 1], (x >> 1) & 1, abort, a.err) ||
              (x > 0 && !mbar_wait_nap(v_done, (x - 1) & 1, abort, a.err)))
            return false;
          tc_fence_after();
          const uint32_t r0k = sw128_desc_lo(smem_u32(smem + Cfg::kR + (x & 1) * 2 * Cfg::kTile), 16);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * Cfg::kChunk + (kk & 3) * 32) >> 4;
            mma_ss(tmem + Cfg::kS, desc_join(f0 + off, dhi), desc_join(r0k + off, dhi), idS, kk > 0);
          }
          mma_commit(s_full);
          return true;
        };
        // Per tile the pipe runs dP^T(g), dV(g), S^T(g + 1), dK(g): the next
        // tile's S^T goes ahead of dK, which waits for the elementwise dS^T.
        ok = mbar_wait_nap(fixed_full, uf & 1, abort, a.err) && issue_s(g);
        for (int i = 0; i < ntot && ok; ++i, ++g) {
          const int sl = g & 1;
          const uint32_t rb = smem_u32(smem + Cfg::kR + sl * 2 * Cfg::kTile);
          const uint32_t r1k = sw128_desc_lo(rb + Cfg::kTile, 16);
          if (g > 0 && !mbar_wait_nap(k_done, (g - 1) & 1, abort, a.err)) { ok = false; break; }
          tc_fence_after();
          // dP^T = V dO^T
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * Cfg::kChunk + (kk & 3) * 32) >> 4;
            mma_ss(tmem + Cfg::kDP, desc_join(f1 + off, dhi), desc_join(r1k + off, dhi), idS, kk > 0);
          }
          mma_commit(dp_full);
          if (i == ntot - 1) mma_commit(fixed_empty);
          // dV += P^T dO (P^T packed over S^T: queries 64h.. at columns 64h..64h+31)
          const uint32_t r0m = sw128_desc_lo(rb, Cfg::kChunk), r1m = sw128_desc_lo(rb + Cfg::kTile, Cfg::kChunk);
          if (!mbar_wait_nap(p_done, g & 1, abort, a.err)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kT / 16; ++kk)
            mma_ts(tmem + Cfg::kDV, tmem + Cfg::kS + 64 * (kk >> 2) + 8 * (kk & 3),
                   desc_join(r1m + kk * ((16 * 128) >> 4), dhi), idAcc, i > 0 || kk > 0);
          mma_commit(v_done);
          if (i + 1 < ntot && !issue_s(g + 1)) { ok = false; break; }
          // dK += dS^T Q (dS^T packed over dP^T the same way)
          if (!mbar_wait_nap(ds_done, g & 1, abort, a.err)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kT / 16; ++kk)
            mma_ts(tmem + Cfg::kDK, tmem + Cfg::kDP + 64 * (kk >> 2) + 8 * (kk & 3),
                   desc_join(r0m + kk * ((16 * 128) >> 4), dhi), idAcc, i > 0 || kk > 0);
          mma_commit(k_done);
          mma_commit(&ring_empty[sl]);
          if (i == ntot - 1) mma_commit(acc_full);
        }
        ++uf;
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      g = __shfl_sync(0xffffffffu, g, 0);
    }
    if (lane == 0) {
      // every MMA issued above has finished before TMEM is released
      mma_commit(mma_done);
      const unsigned long long t0 = global_ns();
      while (!mbar_try_wait(mma_done, 0) && global_ns() - t0 < kWaitTimeoutNs) {}
    }
  } else if (warp < kEwWarps) {
    // ------------------------------------------------------ elementwise ---
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int r = (warp & 3) * 32 + lane;
    const int half = (warp >> 2) & 1;   // which half of the query columns
    const float sl2 = a.scale_log2;
    bool ok = true;
    int g = 0, uf = 0;
    for (int k = 0; ok; ++k) {
      if (!warp_wait(&info_full[k & 1], (k >> 1) & 1, abort, a.err)) { ok = false; break; }
      const int4 in = info[k & 1];
      const int2 kr = rowinfo[(k & 1) * 128 + r];
      warp_arrive(&info_empty[k & 1], lane);
      if (in.x < 0) break;
      const BUnit U = decode<KIND>(a, in.x);
      const int wlo = in.y, ntile = in.z, ntot = ntile * heads;
      const size_t pn = static_cast<size_t>(U.prob) * a.n;
      const bool row_ok = r < U.nrows;
      const int rpos = row_ok ? (kGroup ? a.perm[pn + U.row0 + r] : U.row0 + r) : 0;
      const int klo = kr.x, khi = kr.y;
      const uint64_t sc2 = f2_pack(sl2, sl2);
      for (int i = 0, t = 0; i < ntot; ++i, ++g, t = (t + 1 == ntile ? 0 : t + 1)) {
        if (!kGroup && row_ok && i == max(0, ntot - 3)) {
          // the epilogue's far parts, three tiles ahead so that they are in L2 when read
          const size_t o = (static_cast<size_t>(U.zkv) * a.n + rpos) * D + half * (D / 2);
#pragma unroll
          for (int q = 0; q < D / 2; q += 32) {
            prefetch_l2(a.dv_far + o + q);
            prefetch_l2(a.dk_far + o + q);
          }
        }
        const float* cb = colbuf + (g & 3) * 256;   // [-lse2 x128, -delta x128] of this tile's queries
        const int c0 = wlo + t * kT + half * 64;    // query index of this half's first column
        // bit e: the row keeps column c0 + e
        const int lo = max(klo - c0, 0), hi = min(khi - c0, 63);
        const uint64_t keepm = (row_ok && lo <= hi) ? ((~0ull >> (63 - hi)) & (~0ull << lo)) : 0ull;
        const bool full = __all_sync(0xffffffffu, keepm == ~0ull);
        if (!warp_wait(&col_full[g & 3], (g >> 2) & 1, abort, a.err)) { ok = false; break; }
        if (!warp_wait(s_full, g & 1, abort, a.err)) { ok = false; break; }
        tc_fence_after();
        uint32_t sv[64];
        tmem_ld32(tmem + lane_base + Cfg::kS + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
        tmem_ld32(tmem + lane_base + Cfg::kS + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
        tmem_wait_ld();
        // P = 2^(s scale log2e - lse2) in packed pairs; a dropped pair gets
        // exp2(-inf) = +0, no branch around the exponential
        const uint64_t* nl = reinterpret_cast<const uint64_t*>(cb + half * 64);
        uint64_t p2[32];
        uint32_t pk[32];
        if (full) {
#pragma unroll
          for (int e = 0; e < 64; e += 2) {
            float t0, t1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), sc2, nl[e / 2]), t0, t1);
            const float q0 = ex2f(t0), q1 = ex2f(t1);
            p2[e / 2] = f2_pack(q0, q1);
            pk[e / 2] = pack_bf16x2(q0, q1);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 64; e += 2) {
            float t0, t1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), sc2, nl[e / 2]), t0, t1);
            const float q0 = ex2f((keepm >> e) & 1 ? t0 : -INFINITY);
            const float q1 = ex2f((keepm >> (e + 1)) & 1 ? t1 : -INFINITY);
            p2[e / 2] = f2_pack(q0, q1);
            pk[e / 2] = pack_bf16x2(q0, q1);
          }
        }
        // P^T over the first 32 of this half's 64 S^T columns
        tmem_st32(tmem + lane_base + Cfg::kS + half * 64, pk);
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(p_done, lane);
        if (!warp_wait(dp_full, g & 1, abort, a.err)) { ok = false; break; }
        tc_fence_after();
        // dS = P (dP - Delta) in packed pairs, 32 columns of dP^T at a time
        const uint64_t* nd = reinterpret_cast<const uint64_t*>(cb + 128 + half * 64);
#pragma unroll
        for (int hq = 0; hq < 2; ++hq) {
          uint32_t dv[32];
          tmem_ld32(tmem + lane_base + Cfg::kDP + half * 64 + 32 * hq, dv);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const int q = 16 * hq + e / 2;
            float d0, d1;
            f2_unpack(f2_mul(p2[q], f2_add(f2_pack(__uint_as_float(dv[e]), __uint_as_float(dv[e + 1])), nd[q])), d0, d1);
            pk[q] = pack_bf16x2(d0, d1);
          }
        }
        // dS^T over the first 32 of this half's 64 dP^T columns
        tmem_st32(tmem + lane_base + Cfg::kDP + half * 64, pk);
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(ds_done, lane);
      }
      if (!ok) break;
      // epilogue: this half's dV and dK columns [half * D/2, (half + 1) * D/2)
      const bool have = ntot > 0;
      if (have) {
        if (!warp_wait(acc_full, uf & 1, abort, a.err)) { ok = false; break; }
        ++uf;
        tc_fence_after();
      }
      // Each thread holds its row's values; they go through this warp's 32 x 16
      // fp32 slab in shared memory (16-byte pieces at slot piece ^ ((row >> 1) & 3),
      // so neither the row writes nor the column reads conflict) and leave as
      // 64-byte runs of one row per four lanes.
      float* stg = stage + warp * 512;
      const int jr = lane >> 2, kq = lane & 3;
      const size_t zrow = static_cast<size_t>(U.zkv) * a.n;
      int rp4[4];          // token of pass row 8i + jr
      bool ok4[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        rp4[i] = __shfl_sync(0xffffffffu, rpos, 8 * i + jr);
        ok4[i] = (warp & 3) * 32 + 8 * i + jr < U.nrows;
      }
#pragma unroll
      for (int cm = 0; cm < D / 32; ++cm) {      // (32-column group of this half, dV or dK)
        const int c = half * (D / 64) + (cm >> 1), m = cm & 1;
        const float mul = m ? a.scale : 1.f;     // dK carries the softmax scale
        float* far = m ? a.dk_far : a.dv_far;
        // window kind: the far parts of the group's eight row pieces, in flight
        // while the accumulator is read and staged
        float4 fv[8];
        if (!kGroup) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int i = q & 3, s16 = q >> 2;
            fv[q] = ok4[i] ? *reinterpret_cast<const float4*>(far + (zrow + rp4[i]) * D + c * 32 + s16 * 16 + 4 * kq)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
        uint32_t x[32];
        if (have) {
          tmem_ld32(tmem + lane_base + (m ? Cfg::kDK : Cfg::kDV) + c * 32, x);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) x[e] = 0u;
        }
#pragma unroll
        for (int s16 = 0; s16 < 2; ++s16) {    // 16-column pieces of the 32
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int e = 16 * s16 + 4 * k;
            *reinterpret_cast<float4*>(stg + lane * 16 + 4 * (k ^ ((lane >> 1) & 3))) =
                make_float4(__uint_as_float(x[e]) * mul, __uint_as_float(x[e + 1]) * mul,
                            __uint_as_float(x[e + 2]) * mul, __uint_as_float(x[e + 3]) * mul);
          }
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int j = 8 * i + jr;            // row of this warp's 32
            const float4 v = *reinterpret_cast<const float4*>(stg + j * 16 + 4 * (kq ^ ((j >> 1) & 3)));
            if (ok4[i]) {
              const size_t o = (zrow + rp4[i]) * D + c * 32 + s16 * 16 + 4 * kq;
              if (kGroup) {
                *reinterpret_cast<float4*>(far + o) = v;
              } else {
                const float4 f = fv[4 * s16 + i];
                __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(m ? a.dK : a.dV);
                *reinterpret_cast<uint2*>(dst + o) =
                    make_uint2(pack_bf16x2(v.x + f.x, v.y + f.y), pack_bf16x2(v.z + f.z, v.w + f.w));
              }
            }
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

// The far dK/dV kernel's units (u = kt + nkt * (kv + H_kv * b)) longest first.
// A unit's weight is the number of 128-slot tiles from its first key slot to
// the end of the group of its last one: the query slots that its keys can
// meet lie in that stretch.  One CTA: counting sort over the weights (1 ..
// nkt), units of equal weight in any order (each unit owns its rows, so the
// order changes no result).  Past 12,287 weights it writes the natural order.
__global__ void __launch_bounds__(1024) kv_order_kernel(const BwdArgs a, int n_units) {
  extern __shared__ int cnt[];
  const int nkt = (a.n + kT - 1) / kT;
  const int nb = nkt + 1;
  if (nb > 12287) {
    for (int u = threadIdx.x; u < n_units; u += blockDim.x) a.kv_order[u] = u;
    return;
  }
  auto weight = [&](int u) {
    const int kt = u % nkt, r = u / nkt;
    const int kv = r % a.H_kv, b = r / a.H_kv;
    const int32_t* off = a.offsets + static_cast<size_t>(b * a.A + (a.A == 1 ? 0 : kv)) * (a.groups + 1);
    const int row0 = kt * kT, last = min(a.n, row0 + kT) - 1;
    int lo = 0, hi = a.groups;   // off[lo] <= last < off[lo + 1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (off[mid] <= last) lo = mid; else hi = mid;
    }
    return min(nkt, max(1, (off[lo + 1] - row0 + kT - 1) / kT));
  };
  for (int i = threadIdx.x; i < nb; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  for (int u = threadIdx.x; u < n_units; u += blockDim.x) atomicAdd(&cnt[weight(u)], 1);
  __syncthreads();
  if (threadIdx.x == 0) {   // first position of each weight, heaviest first
    int run = 0;
    for (int w = nb - 1; w >= 0; --w) {
      const int c = cnt[w];
      cnt[w] = run;
      run += c;
    }
  }
  __syncthreads();
  for (int u = threadIdx.x; u < n_units; u += blockDim.x) a.kv_order[atomicAdd(&cnt[weight(u)], 1)] = u;
}

// Q, dO rows and the LSE of every query head in the order of its assignment's
// index, dst[zq, s] = src[zq, perm_a[s]] (a = the head's assignment), and
// Delta_i = dO_i . O_i (fp32) of every row in both orders.  d / 8 lanes per
// row, 16 bytes each; the lanes of a row are an aligned group of the warp and
// every lane of a warp runs every iteration, so the row's shuffle reduction
// always sees the whole warp.
__global__ void __launch_bounds__(256) permute_q_kernel(BwdArgs a, __nv_bfloat16* Qs, __nv_bfloat16* dOs,
                                                        float* lse_s, float* delta_s, long long total) {
  const int vpr = a.d / 8;
  const int lane = lane_id();
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long base = blockIdx.x * static_cast<long long>(blockDim.x) + (threadIdx.x & ~31u); base < total;
       base += stride) {
    const long long e = base + lane;
    const bool act = e < total;
    float dsum = 0.f;
    long long row = 0, src = 0;
    int u = 0;
    if (act) {
      row = e / vpr;
      u = static_cast<int>(e % vpr);
      const int s = static_cast<int>(row % a.n);
      const long long zq = row / a.n;
      const int h = static_cast<int>(zq % a.H);
      const long long b = zq / a.H;
      const long long p = b * a.A + (a.A == 1 ? 0 : (h * a.H_kv) / a.H);
      src = zq * a.n + __ldg(a.perm + p * a.n + s);
      const uint4 q = __ldg(reinterpret_cast<const uint4*>(a.Q) + src * vpr + u);
      const uint4 g = __ldg(reinterpret_cast<const uint4*>(a.dO) + src * vpr + u);
      const uint4 o = __ldg(reinterpret_cast<const uint4*>(a.O) + src * vpr + u);
      reinterpret_cast<uint4*>(Qs)[e] = q;
      reinterpret_cast<uint4*>(dOs)[e] = g;
      const uint32_t gw[4] = {g.x, g.y, g.z, g.w}, ow[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        dsum = fmaf(__uint_as_float(gw[j] << 16), __uint_as_float(ow[j] << 16), dsum);
        dsum = fmaf(__uint_as_float(gw[j] & 0xffff0000u), __uint_as_float(ow[j] & 0xffff0000u), dsum);
      }
    }
    for (int off = vpr >> 1; off > 0; off >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, off);
    if (act && u == 0) {
      lse_s[row] = a.lse[src];
      delta_s[row] = dsum;
      a.delta[src] = dsum;
    }
  }
}

template <int D>
cudaError_t launch_d(const BwdArgs& a, const CUtensorMap* qs, const CUtensorMap* dos, const CUtensorMap* ks,
                     const CUtensorMap* vs, const CUtensorMap* q3, const CUtensorMap* do3, const CUtensorMap* k3,
                     const CUtensorMap* v3, int max_items, int num_sms, cudaStream_t st) {
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
  const unsigned kv_grid = static_cast<unsigned>(std::min(k_units, sms));
  const int nb = (a.n + kT - 1) / kT + 1;
  kv_order_kernel<<<1, 1024, nb <= 12287 ? nb * 4 : 0, st>>>(a, static_cast<int>(k_units));
  bwd_dkv_kernel<D, kDkvGroup><<<kv_grid, kThreads, KvCfg<D>::kSmem, st>>>(*qs, *dos, *ks, *vs, a);
  bwd_dkv_kernel<D, kDkvLocal><<<kv_grid, kThreads, KvCfg<D>::kSmem, st>>>(*q3, *do3, *k3, *v3, a);
  return cudaGetLastError();
}

template <int D>
cudaError_t set_smem_d() {
  cudaError_t e;
  e = cudaFuncSetAttribute(bwd_dq_kernel<D, kDqGroup>, cudaFuncAttributeMaxDynamicSharedMemorySize, DqCfg<D>::kSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(bwd_dq_kernel<D, kDqLocal>, cudaFuncAttributeMaxDynamicSharedMemorySize, DqCfg<D>::kSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(bwd_dkv_kernel<D, kDkvGroup>, cudaFuncAttributeMaxDynamicSharedMemorySize, KvCfg<D>::kSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(bwd_dkv_kernel<D, kDkvLocal>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              KvCfg<D>::kSmem);
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
