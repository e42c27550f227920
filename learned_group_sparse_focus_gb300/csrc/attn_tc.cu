// Focus attention on the tcgen05 tensor cores (bf16 in, fp32 accumulate).
//
// "Focus: Learning Which Attention Pairs Matter", section 2.1: local window
// pairs at full resolution, far pairs only inside a group; section 2.2: far
// pairs of different groups are skipped outright; section 3.3 and "Why Attend
// to Everything? Focus is the Key", section 2.3: the pattern splits into a
// local-window attention and an in-group causal attention whose softmaxes
// combine exactly ("Why Attend to Everything?", section 2.1).
//
// One persistent kernel, three modes; a work unit is one 128-row query tile:
//   group  a work item: <= 128 sorted slots of one group; keys are the group's
//          earlier members at or before i - w (slot < farlen of the row), read
//          from K/V pre-permuted into sorted order so each key tile is one
//          dense TMA box.  Writes the normalised partial O and its LSE at each
//          row's item (its token position, or with top-k membership its entry
//          i * k + c, whose query is token i).
//   local  128 consecutive tokens, keys j in [i - w + 1, i]; merges the group
//          partial by log-sum-exp when the row has far keys; writes O.
//   dense  128 consecutive tokens, keys j in [i - w + 1, i] and no partial:
//          plain causal attention with w = n (the comparator), a standalone
//          sliding-window call with the Focus window.
//
// S = Q K^T reads Q and K from shared memory; O += P V reads P from TMEM and
// V from shared memory.  TMEM (512 columns for d = 128): three S buffers of
// 128 columns and O (d columns).  The softmax writes P(t) as bf16 pairs over
// the S(t) it has just read, so a buffer is free again once O += P(t) V(t) is
// done: the S products of the next two tiles run while the softmax works, and
// the softmax never waits for the PV product of the tile before.
//
// Warp roles (384 threads), one CTA per SM looping over units:
//   warps 0-7   softmax, two warps per query row (warps w and w + 4 share TMEM
//               lane quadrant w, each takes half of every row's columns): per
//               key tile read the half S row from TMEM, apply the keep rule to
//               boundary tiles, agree on the row max with the partner through
//               shared memory, exp2 and sum in fp32, write the half P row,
//               rescale the half O row only when the running max grows by
//               more than 2^8; the epilogue of a unit runs at the start of the
//               next one, so the next unit's first S products overlap it: it
//               builds the O tile in shared memory (in the local pass merged
//               with the group partial the V load warp staged there) for the V
//               load warp to store
//   warp 8      Q tiles into a 2-slot ring and K tiles into a 2-slot ring
//               (TMA; a TMA row gather through perm for the group pass's Q)
//   warp 9      TMEM owner; issues O += P(t) V(t) once P(t) is written
//   warp 10     issues S(t) = Q K(t)^T once the softmax has read S(t-2),
//               the previous content of the same buffer
//   warp 11     V tiles into a 2-slot ring; it also stores each unit's O tile
//               from the stage with TMA (a tile::scatter4 row scatter to the
//               token positions in the group pass) and then (local) loads the
//               next unit's group-partial tile into the stage
// The load and MMA warps wait by polling with short sleeps: an issuing thread
// that spins, or a tcgen05.mma queued behind a busy tensor pipe, slows the
// softmax warps that share its SM sub-partition.
// Every wait is bounded; on timeout the CTA raises an error bit, drains its
// copies, frees TMEM and exits.
#include "common.cuh"
#include "kernels.h"

namespace focus {
namespace {

constexpr int kBN = 128;                     // keys per tile
constexpr int kBM = 128;                     // query rows per unit
constexpr float kRescaleThreshold = 8.0f;    // log2 units
constexpr int kSoftmaxWarps = 8;            // two per TMEM lane quadrant
constexpr int kWarpLoad = kSoftmaxWarps;     // TMA loads
constexpr int kWarpPV = kSoftmaxWarps + 1;   // TMEM owner, O += P V issuer
constexpr int kWarpS = kSoftmaxWarps + 2;    // S = Q K^T issuer
constexpr int kWarpLoadV = kSoftmaxWarps + 3;  // V tiles (and the group partial)
constexpr int kThreads = 32 * (kSoftmaxWarps + 4);
// Register split (setmaxnreg).  The kernel launches at 168 registers per thread
// (384 x 168 = 64512, the cap for 12 warps).  Warpgroup 2 gives registers back
// down to 88 and the two softmax warpgroups take them up to 208:
// 128 * 88 + 256 * 208 = 64512, and each SM sub-partition then holds
// 208 + 208 + 88 = 504 registers per lane (<= 512).
constexpr int kRegsLow = 88;
constexpr int kRegsHigh = 208;
// Three rings of tile slots.  Q tiles (one per unit, read by every S product
// of the unit) get two slots, so the next unit's Q lands while this unit runs.
// K slots are free once their S product is done, early in a tile's life; V
// slots only once O += P V is, late in it.  Separate rings keep a slow V from
// holding up the next K.
constexpr int kQSlots = 2;
constexpr int kKSlots = 2;
constexpr int kVSlots = 2;
// S buffers in TMEM.  The softmax writes P(g) as bf16 pairs over the S(g) it
// has just read (each half-row warp into the first 32 columns of its own 64),
// so a buffer is free again once O += P(g) V(g) is done, and no P buffer of its
// own has to be waited for before the write.
constexpr int kSBuf = 3;

template <int D>
struct AttnCfg {
  static constexpr int kChunk = 128 * 128;   // 64 columns x 128 rows, one swizzle slab
  static constexpr int kTile = 128 * D * 2;  // one 128-row Q/K/V tile
  static constexpr int kQ = 0;                            // Q ring
  static constexpr int kK = kQ + kQSlots * kTile;         // K ring
  static constexpr int kV = kK + kKSlots * kTile;         // V ring
  static constexpr int kOst = kV + kVSlots * kTile;       // O tile staging
  static constexpr int kBar = kOst + kTile;                 // barriers (< 256 B)
  static constexpr int kXch = kBar + 256;                   // row max / sum exchange: [2][2][128] fp32
  static constexpr int kRowTok = kXch + 2 * 2 * 128 * 4;    // group pass: O_far row of each tile row
  static constexpr int kSmem = kRowTok + 128 * 4;
  static constexpr uint32_t kS = 0;          // kSBuf S buffers of 128 columns (P over S)
  static constexpr uint32_t kO = kSBuf * 128;  // O: d columns
  static constexpr uint32_t kTmemCols = 512;
};

static_assert(AttnCfg<128>::kSmem <= 227 * 1024, "attention shared memory above the 227 KB per CTA");
static_assert(AttnCfg<128>::kO + 128 <= AttnCfg<128>::kTmemCols, "S buffers and O exceed TMEM");
static_assert(kBN / 2 % 16 == 0, "the half-row max walks 16 columns per step");

// max(a, b, c) in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// One arrival per warp: the lanes' earlier work (TMEM reads and writes, shared
// memory stores, each already fenced by its own lane) is ordered before lane
// 0's arrival by the warp barrier.
__device__ __forceinline__ void warp_arrive(uint64_t* bar, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

// warp-uniform bounded wait (every lane waits; the outcome is shared)
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          int* err, unsigned long long limit_ns) {
  const bool ok = mbar_wait(bar, parity, abort, err, limit_ns);
  return __all_sync(0xffffffffu, ok);
}

struct Unit {
  int b, h, prob, zkv, zq, ybase;
  int row0, nrows;
  int t0, t1;   // inclusive key-tile range
  int sub;      // group pass over a split top-2 index: the key sub-run's column
  int grp;      // split index: the rows' group g (virtual group v = g * K + o)
};

// Split top-2 index: a unit's keys are the sub-runs (g, o') of its group in
// increasing o' (column j = o' - (o' > g)), each up to the far prefix of the
// unit's last row; empty ones are skipped.  The walk gives, tile by tile, the
// column, the tile within it and the sub-run's first slot.
// sub-run columns per split unit (K <= 8)
constexpr int kMaxSub = 7;

// a[j] for a runtime j < kMaxSub, without local memory
__device__ __forceinline__ int pick(const int (&a)[kMaxSub], int j) {
  int v = a[0];
#pragma unroll
  for (int q = 1; q < kMaxSub; ++q) v = q == j ? a[q] : v;
  return v;
}

struct SegWalk {
  int j, tt, nt, key0;
  __device__ __forceinline__ void next_col(const AttnArgs& a, const Unit& U) {
    const int K = a.nsub + 1;
    const int32_t* last = a.farlen_sub + (static_cast<size_t>(U.prob) * a.m + U.row0 + U.nrows - 1) * a.nsub;
    for (++j; j < a.nsub; ++j) {
      const int keys = last[j];
      if (keys > 0) {
        const int o2 = j < U.grp ? j : j + 1;
        nt = (keys + kBN - 1) / kBN;
        tt = 0;
        key0 = a.offsets[static_cast<size_t>(U.prob) * (K * K + 1) + U.grp * K + o2];
        return;
      }
    }
  }
  __device__ __forceinline__ void begin(const AttnArgs& a, const Unit& U) {
    j = -1;
    next_col(a, U);
  }
  // true when the next tile starts a new column
  __device__ __forceinline__ bool step(const AttnArgs& a, const Unit& U) {
    if (++tt < nt) return false;
    next_col(a, U);
    return true;
  }
};

template <int MODE>
__device__ __forceinline__ int unit_count(const AttnArgs& a) {
  if (is_group_mode(MODE)) {
    const int hpa = a.A == 1 ? a.H : a.H / a.H_kv;
    return *a.n_items * hpa;
  }
  return a.B * a.H * ((a.n + kBM - 1) / kBM);
}

template <int MODE>
__device__ __forceinline__ void decode_unit(const AttnArgs& a, int u, const focus_item_t& it, Unit& U) {
  int kv, asg;
  if (is_group_mode(MODE)) {
    const int hpa = a.A == 1 ? a.H : a.H / a.H_kv;
    const int y = u % hpa;
    U.b = it.b;
    asg = it.a;
    U.h = a.A == 1 ? y : it.a * (a.H / a.H_kv) + y;
    kv = (U.h * a.H_kv) / a.H;
    U.row0 = it.row0;
    U.nrows = it.rows;
    U.t0 = 0;
    U.t1 = (it.keys + kBN - 1) / kBN - 1;
    U.ybase = it.key0;
    U.sub = it.pad;
    U.grp = 0;
    if (MODE == kModeGroupSplit) {
      // tiles = the sub-runs' tiles, each rounded up on its own
      const int K = a.nsub + 1;
      U.grp = it.g / K;
      const int32_t* last = a.farlen_sub +
                            (static_cast<size_t>(it.b * a.A + it.a) * a.m + it.row0 + it.rows - 1) * a.nsub;
      int nt = 0;
      for (int j = 0; j < a.nsub; ++j) nt += (last[j] + kBN - 1) / kBN;
      U.t1 = nt - 1;
    }
  } else {
    U.h = u % a.H;
    const int r = u / a.H;
    const int nqt = (a.n + kBM - 1) / kBM;
    const int qt = nqt - 1 - (r % nqt);          // longest units first
    U.b = r / nqt;
    kv = (U.h * a.H_kv) / a.H;
    asg = a.A == 1 ? 0 : kv;
    U.row0 = qt * kBM;
    U.nrows = min(kBM, a.n - U.row0);
    U.t0 = max(0, U.row0 - a.w + 1) / kBN;
    U.t1 = (U.row0 + U.nrows - 1) / kBN;
    U.ybase = 0;
    U.sub = 0;
    U.grp = 0;
  }
  U.prob = U.b * a.A + asg;
  U.zkv = U.b * a.H_kv + kv;
  U.zq = U.b * a.H + U.h;
}

// Unit walked by this CTA in round k, or -1 past the end.  Rounds alternate
// direction (0..G-1, then G-1..0, ...), so over a longest-first unit list
// every CTA gets a balanced mix of long and short units.
__device__ __forceinline__ int snake_unit(int k, int n_units) {
  const int G = gridDim.x, base = k * G;
  if (base >= n_units) return -1;
  const int u = base + ((k & 1) ? G - 1 - static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x));
  return u < n_units ? u : -2;
}

// Every role walks the same units.  In the group pass a unit is named by two
// dependent loads (its order entry, then its item); the walk keeps the next
// round's item and the order entry of the round after it in flight while the
// current unit runs, so neither load sits on a role's path at a unit boundary.
template <int MODE>
struct UnitWalk {
  focus_item_t nxt;   // item of round k + 1's unit
  int ord;            // order entry of round k + 2's unit
  int hpa, n_units;

  __device__ __forceinline__ void begin(const AttnArgs& a, int n) {
    n_units = n;
    hpa = a.A == 1 ? a.H : a.H / a.H_kv;
    if (is_group_mode(MODE)) {
      const int u0 = snake_unit(0, n), u1 = snake_unit(1, n);
      if (u0 >= 0) nxt = a.items[a.order[u0 / hpa]];
      ord = u1 >= 0 ? a.order[u1 / hpa] : 0;
    }
  }
  // Round k's unit (as snake_unit: -1 past the end, -2 none this round),
  // decoded into U when there is one.
  __device__ __forceinline__ int step(const AttnArgs& a, int k, Unit& U) {
    const int u = snake_unit(k, n_units);
    if (is_group_mode(MODE)) {
      const focus_item_t it = nxt;
      if (snake_unit(k + 1, n_units) >= 0) nxt = a.items[ord];
      const int u2 = snake_unit(k + 2, n_units);
      if (u2 >= 0) ord = a.order[u2 / hpa];
      if (u >= 0) decode_unit<MODE>(a, u, it, U);
    } else if (u >= 0) {
      decode_unit<MODE>(a, u, nxt, U);
    }
    return u;
  }
};

// What the epilogue of a unit needs once its tile loop is over.  In the local
// pass the row's far flag and group LSE are read when the unit starts (and its
// group O row is prefetched into L2), so their latency hides behind the tiles.
struct RowState {
  int pos, prob, zq, row0;
  bool valid, far;
  float m, l, lse_far;
};

template <int D, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                   const __grid_constant__ CUtensorMap tm_of, const AttnArgs a) {
  using Cfg = AttnCfg<D>;
  constexpr int kChunks = D / 64;

  // The layout uses the whole 227 KB, with no room to realign: the dynamic
  // shared memory base must already sit on a 1024-byte boundary (the 128-byte
  // swizzle atoms), which it does when the kernel declares no static shared
  // memory.  Checked, not assumed: a misaligned base only raises an error.
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) atomicOr(a.err, kErrInternal);
    return;
  }
  uint8_t* smem = smem_raw;
  uint8_t* sQ = smem + Cfg::kQ;
  uint8_t* sK = smem + Cfg::kK;
  uint8_t* sV = smem + Cfg::kV;
  uint8_t* sO = smem + Cfg::kOst;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kBar);
  uint64_t* pv_done = bars + 0;       // [kSBuf] per S buffer: O += P V from it done
  uint64_t* o_final = pv_done + kSBuf;  // one phase per unit: its last PV landed
  uint64_t* o_free = o_final + 1;     // one phase per unit: O read out (softmax warps)
  uint64_t* s_full = o_free + 1;      // [kSBuf] per S buffer
  uint64_t* p_ready = s_full + kSBuf; // [kSBuf] per S buffer: P written over S (softmax warps)
  uint64_t* ofar_full = p_ready + kSBuf;  // local: the unit's group-partial tile is staged
  uint64_t* ost_free = ofar_full + 1; // group, dense: the O stage was stored out (1 arrival)
  uint64_t* ost_full = ost_free + 1;  // local/dense: the O stage is written (softmax warps)
  uint64_t* q_full = ost_full + 1;    // [kQSlots]
  uint64_t* q_empty = q_full + kQSlots;
  uint64_t* k_full = q_empty + kQSlots;   // [kKSlots]
  uint64_t* k_empty = k_full + kKSlots;
  uint64_t* v_full = k_empty + kKSlots;   // [kVSlots]
  uint64_t* v_empty = v_full + kVSlots;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(v_empty + kVSlots);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* xch = reinterpret_cast<float*>(smem + Cfg::kXch);
  int* row_tok = reinterpret_cast<int*>(smem + Cfg::kRowTok);

  const int warp = warp_id(), lane = lane_id();
  const int n_units = unit_count<MODE>(a);
  if (threadIdx.x == 0) {
    mbar_init(o_final, 1);
    mbar_init(o_free, kSoftmaxWarps);
    mbar_init(ofar_full, 1);
    mbar_init(ost_free, 1);
    mbar_init(ost_full, kSoftmaxWarps);
    for (int x = 0; x < kSBuf; ++x) {
      mbar_init(&pv_done[x], 1);
      mbar_init(&s_full[x], 1);
      mbar_init(&p_ready[x], kSoftmaxWarps);
    }
    for (int k = 0; k < kQSlots; ++k) {
      mbar_init(&q_full[k], 1);
      mbar_init(&q_empty[k], 1);
    }
    for (int k = 0; k < kKSlots; ++k) {
      mbar_init(&k_full[k], 1);
      mbar_init(&k_empty[k], 1);
    }
    for (int k = 0; k < kVSlots; ++k) {
      mbar_init(&v_full[k], 1);
      mbar_init(&v_empty[k], 1);
    }
    *abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_o);
    if (MODE == kModeLocal) prefetch_tmap(&tm_of);
  }
  if (warp == kWarpPV) tmem_alloc(tmem_slot, Cfg::kTmemCols);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= kSoftmaxWarps) {
    // warpgroup 2 (the two load warps and the two MMA issuers) hands registers
    // to the softmax warpgroups
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
    if (warp == kWarpLoad) {
      // -------------------------------------------------- Q and K loads ---
      int qn = 0;                // Q tiles requested in full
      int ck = 0;                // K tiles issued
      bool ok = true;
      UnitWalk<MODE> walk;
      walk.begin(a, n_units);
      // Group passes: a unit's Q tile is 128 row gathers through perm (lane l:
      // rows 4l..4l+3 of every 64-column slab).  The next unit's gathers go
      // out in kQBatches batches (lanes 4j..4j+3, 8 gathers each) between this
      // unit's K loads, one batch per K tile once the Q slot is free, so the
      // tile is in place when the unit's first S product is due and no long
      // run of gathers sits in front of a K load in the SM's TMA queue (4 or
      // 16 batches measured slower than 8).
      constexpr int kQBatches = 8;
      Unit U_nx;
      int u_nx = -1, nx_b = 0, rows_nx[4] = {0, 0, 0, 0};
      bool have_nx = false;
      auto gather_rows = [&](const Unit& V, int (&rows)[4]) {
        // rows past the item repeat its first row, whose scores are all masked
        const int32_t* pp = a.perm + static_cast<size_t>(V.prob) * a.m + V.row0;
        const int first = pp[0] >> a.kshift;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int rr = 4 * lane + j;
          rows[j] = V.zq * a.n + (rr < V.nrows ? pp[rr] >> a.kshift : first);
        }
      };
      // batch bt of Q tile qn (its slot already free)
      auto q_batch = [&](const int (&rows)[4], int bt) {
        const int sl = qn % kQSlots;
        if (bt == 0) {
          if (lane == 0) mbar_expect_tx(&q_full[sl], Cfg::kTile);
          __syncwarp();
        }
        if (lane / (32 / kQBatches) == bt) {
          uint8_t* dst = sQ + sl * Cfg::kTile;
#pragma unroll
          for (int ch = 0; ch < kChunks; ++ch)
            tma_gather4(dst + ch * Cfg::kChunk + 4 * lane * 128, &tm_q, &q_full[sl], ch * 64, rows[0], rows[1],
                        rows[2], rows[3]);
        }
      };
      for (int k = 0; ok; ++k) {
        Unit U;
        int u, rows[4] = {0, 0, 0, 0}, done_b = 0;
        if (have_nx) {
          have_nx = false;
          u = u_nx;
          U = U_nx;
          done_b = nx_b;
#pragma unroll
          for (int j = 0; j < 4; ++j) rows[j] = rows_nx[j];
        } else {
          u = walk.step(a, k, U);
          if (is_group_mode(MODE) && u >= 0) gather_rows(U, rows);
        }
        if (u == -1) break;
        if (u < 0) continue;
        {
          // the unit's Q tile (group passes: the batches its predecessor did not issue)
          const int sl = qn % kQSlots, use = qn / kQSlots;
          bool qf = true;
          if (lane == 0 && done_b == 0 && use > 0) qf = mbar_wait_nap(&q_empty[sl], (use - 1) & 1, abort, a.err, a.wait_ns);
          if (!__shfl_sync(0xffffffffu, qf ? 1 : 0, 0)) break;
          uint8_t* dst = sQ + sl * Cfg::kTile;
          if (a.hold_first_q && qn == 0) {
            // test hook: this tile is never requested, so its wait runs out
          } else if (is_group_mode(MODE)) {
            for (int bt = done_b; bt < kQBatches; ++bt) q_batch(rows, bt);
          } else if (lane == 0) {
            mbar_expect_tx(&q_full[sl], Cfg::kTile);
#pragma unroll
            for (int ch = 0; ch < kChunks; ++ch)
              tma_load_3d(dst + ch * Cfg::kChunk, &tm_q, &q_full[sl], ch * 64, U.row0, U.zq);
          }
          ++qn;
        }
        if (is_group_mode(MODE)) {
          // the next unit, named one walk round early
          u_nx = walk.step(a, k + 1, U_nx);
          have_nx = true;
          nx_b = 0;
          if (u_nx >= 0) gather_rows(U_nx, rows_nx);
        }
        SegWalk sw;
        if (MODE == kModeGroupSplit) sw.begin(a, U);
        for (int t = U.t0; t <= U.t1; ++t, ++ck) {
          if (is_group_mode(MODE) && u_nx >= 0 && nx_b < kQBatches) {
            // one batch of the next unit's Q, if its slot is free (lane 0's view)
            const int qsl = qn % kQSlots, quse = qn / kQSlots;
            const bool fr = quse == 0 || mbar_test_wait(&q_empty[qsl], (quse - 1) & 1);
            if (__shfl_sync(0xffffffffu, fr ? 1 : 0, 0)) q_batch(rows_nx, nx_b++);
          }
          const int sl = ck % kKSlots, use = ck / kKSlots;
          // lane 0 polls; the other lanes wait at the shuffle without issuing
          bool kf = true;
          if (lane == 0 && use > 0) kf = mbar_wait_nap(&k_empty[sl], (use - 1) & 1, abort, a.err, a.wait_ns);
          if (!__shfl_sync(0xffffffffu, kf ? 1 : 0, 0)) { ok = false; break; }
          const int krow = MODE == kModeGroupSplit ? sw.key0 + sw.tt * kBN : U.ybase + t * kBN;
          if (lane == 0) {
            mbar_expect_tx(&k_full[sl], Cfg::kTile);
#pragma unroll
            for (int ch = 0; ch < kChunks; ++ch)
              tma_load_3d(sK + sl * Cfg::kTile + ch * Cfg::kChunk, &tm_k, &k_full[sl], ch * 64, krow, U.zkv);
          }
          if (MODE == kModeGroupSplit) sw.step(a, U);
        }
        ok = __shfl_sync(0xffffffffu, (ok && !*abort) ? 1 : 0, 0) != 0;   // one view for the warp
      }
      if (is_group_mode(MODE) && have_nx && u_nx >= 0 && nx_b > 0) {
        // stopped with a tile part-requested: request the rest (its slot is
        // free) so that the whole tile lands and the drain below can wait for it
        for (int bt = nx_b; bt < kQBatches; ++bt) q_batch(rows_nx, bt);
        ++qn;
      }
      if (*abort && lane == 0) {
        // drain: TMA copies already issued must land before the CTA exits
        for (int L = max(0, ck - kKSlots); L < ck; ++L) {
          const unsigned long long t0 = global_ns();
          while (!mbar_try_wait(&k_full[L % kKSlots], (L / kKSlots) & 1) &&
                 global_ns() - t0 < a.wait_ns) {}
        }
        for (int L = max(a.hold_first_q ? 1 : 0, qn - kQSlots); L < qn; ++L) {
          const unsigned long long t0 = global_ns();
          while (!mbar_try_wait(&q_full[L % kQSlots], (L / kQSlots) & 1) &&
                 global_ns() - t0 < a.wait_ns) {}
        }
      }
    } else if (warp == kWarpLoadV) {
      // ------------------------- V loads; O stage out and group partial in ---
      // This thread also owns the O stage: once the softmax warps have written
      // a unit's O tile there (ost_full) it stores the tile with TMA (in the
      // group pass scattered row by row to the token positions) and, when the
      // copy has read the stage, loads the next unit's group partial into it
      // (local) or releases it (group, dense).
      if (lane == 0) {
        int cv = 0;              // V ring entries issued
        int un = 0;              // units walked
        int ofn = 0;             // group-partial tiles issued
        bool ok = true;
        int prow0 = 0, pzq = 0;  // the previous unit's tile
        auto store_prev = [&]() -> bool {
          if (!mbar_wait_nap(ost_full, (un - 1) & 1, abort, a.err, a.wait_ns)) return false;
          if (is_group_mode(MODE)) {
            // four rows per scatter, one 64-column slab at a time
#pragma unroll 4
            for (int q4 = 0; q4 < 32; ++q4) {
              const int4 rt = *reinterpret_cast<const int4*>(row_tok + 4 * q4);
#pragma unroll
              for (int ch = 0; ch < kChunks; ++ch)
                tma_scatter4(&tm_o, sO + ch * Cfg::kChunk + 4 * q4 * 128, ch * 64, rt.x, rt.y, rt.z, rt.w);
            }
          } else {
            // rows past n fall outside the tensor map and are not written
#pragma unroll
            for (int ch = 0; ch < kChunks; ++ch) tma_store_3d(&tm_o, sO + ch * Cfg::kChunk, ch * 64, prow0, pzq);
          }
          tma_store_commit();
          tma_store_wait_read();
          if (MODE != kModeLocal) mbar_arrive(ost_free);
          return true;
        };
        UnitWalk<MODE> walk;
        walk.begin(a, n_units);
        for (int k = 0; ok; ++k) {
          Unit U;
          const int u = walk.step(a, k, U);
          if (u == -1) break;
          if (u < 0) continue;
          SegWalk sw;
          if (MODE == kModeGroupSplit) sw.begin(a, U);
          for (int t = U.t0, i = 0; t <= U.t1; ++t, ++cv, ++i) {
            const int sl = cv % kVSlots, use = cv / kVSlots;
            if (use > 0 && !mbar_wait_nap(&v_empty[sl], (use - 1) & 1, abort, a.err, a.wait_ns)) { ok = false; break; }
            const int vrow = MODE == kModeGroupSplit ? sw.key0 + sw.tt * kBN : U.ybase + t * kBN;
            mbar_expect_tx(&v_full[sl], Cfg::kTile);
#pragma unroll
            for (int ch = 0; ch < kChunks; ++ch)
              tma_load_3d(sV + sl * Cfg::kTile + ch * Cfg::kChunk, &tm_v, &v_full[sl], ch * 64, vrow, U.zkv);
            if (MODE == kModeGroupSplit) sw.step(a, U);
            // after this unit's first V tiles: the previous unit's O, whose
            // epilogue runs at the start of this unit, then this unit's partial
            if (i == min(1, U.t1 - U.t0)) {
              if (un > 0 && !store_prev()) { ok = false; break; }
              if (MODE == kModeLocal) {
                mbar_expect_tx(ofar_full, Cfg::kTile);
#pragma unroll
                for (int ch = 0; ch < kChunks; ++ch)
                  tma_load_3d(sO + ch * Cfg::kChunk, &tm_of, ofar_full, ch * 64, U.row0, U.zq);
                ++ofn;
              }
            }
          }
          prow0 = U.row0;
          pzq = U.zq;
          ++un;
          ok = ok && !*abort;
        }
        if (ok && un > 0) {
          ok = store_prev();
          tma_store_wait_all();
        }
        if (*abort || !ok) {
          // drain: copies already issued must land before the CTA exits
          tma_store_wait_all();
          for (int L = max(0, cv - kVSlots); L < cv; ++L) {
            const unsigned long long t0 = global_ns();
            while (!mbar_try_wait(&v_full[L % kVSlots], (L / kVSlots) & 1) &&
                   global_ns() - t0 < a.wait_ns) {}
          }
          if (ofn > 0) {
            const unsigned long long t0 = global_ns();
            while (!mbar_try_wait(ofar_full, (ofn - 1) & 1) && global_ns() - t0 < a.wait_ns) {}
          }
        }
      }
    } else if (warp == kWarpPV || warp == kWarpS) {
      // ----------------------------------------------------------- MMAs ---
      // Two issuing threads: one warp issues the S products, the other the PV
      // products.  The two chains share no TMEM (S buffers and Q vs P and O), so
      // neither waits on the other's barriers and the tensor pipe sees both.
      if (lane == 0) {
        constexpr uint32_t idS = idesc_bf16_f32(128, kBN, false, false);
        constexpr uint32_t idPV = idesc_bf16_f32(128, D, false, true);
        constexpr uint32_t dhi = sw128_desc_hi();
        const uint32_t klo = sw128_desc_lo(smem_u32(sK), 16);           // K slots, K-major
        const uint32_t vlo = sw128_desc_lo(smem_u32(sV), Cfg::kChunk);  // V slots, MN-major
        int g = 0;        // tiles (S buffers) walked
        int ck = 0;       // K ring entries walked
        int cv = 0;       // V ring entries walked
        int un = 0;       // units walked
        bool ok = true;
        UnitWalk<MODE> walk;
        walk.begin(a, n_units);
        for (int k = 0; ok; ++k) {
          Unit U;
          const int u = walk.step(a, k, U);
          if (u == -1) break;
          if (u < 0) continue;
          const int nt = U.t1 - U.t0 + 1;
          if (warp == kWarpS) {
            // S(gg) = Q K^T into S buffer gg % kSBuf once O += P(gg-kSBuf) V is
            // done (P lies over the buffer's previous S); the unit's Q slot is
            // released after its last S product
            const int qsl = un % kQSlots;
            if (!mbar_wait_nap(&q_full[qsl], (un / kQSlots) & 1, abort, a.err, a.wait_ns)) break;
            const uint32_t q0 = sw128_desc_lo(smem_u32(sQ + qsl * Cfg::kTile), 16);
            for (int i = 0; i < nt; ++i, ++ck) {
              const int gg = g + i;
              const int sb = gg % kSBuf;
              if (gg >= kSBuf && !mbar_wait_nap(&pv_done[sb], (gg / kSBuf - 1) & 1, abort, a.err, a.wait_ns)) { ok = false; break; }
              const int sl = ck % kKSlots;
              if (!mbar_wait_nap(&k_full[sl], (ck / kKSlots) & 1, abort, a.err, a.wait_ns)) { ok = false; break; }
              tc_fence_after();
              const uint32_t b0 = klo + sl * (Cfg::kTile >> 4);
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = ((kk >> 2) * Cfg::kChunk + (kk & 3) * 32) >> 4;
                mma_ss(tmem + Cfg::kS + 128 * sb, desc_join(q0 + off, dhi), desc_join(b0 + off, dhi),
                       idS, kk > 0);
              }
              mma_commit(&s_full[sb]);
              mma_commit(&k_empty[sl]);
            }
            if (!ok) break;
            mma_commit(&q_empty[qsl]);
          } else {
            // O += P(gg) V(gg)
            for (int i = 0; i < nt; ++i, ++cv) {
              const int gg = g + i;
              const int sl = cv % kVSlots;
              if (!mbar_wait_nap(&v_full[sl], (cv / kVSlots) & 1, abort, a.err, a.wait_ns)) { ok = false; break; }
              if (i == 0 && un > 0 && !mbar_wait_nap(o_free, (un - 1) & 1, abort, a.err, a.wait_ns)) { ok = false; break; }
              const int sb = gg % kSBuf;
              if (!mbar_wait_nap(&p_ready[sb], (gg / kSBuf) & 1, abort, a.err, a.wait_ns)) { ok = false; break; }
              tc_fence_after();
              const uint32_t vb = vlo + sl * (Cfg::kTile >> 4);
#pragma unroll
              for (int kk = 0; kk < kBN / 16; ++kk)
                // keys 16kk..16kk+15 of P(gg): half kk / 4 of the row, packed
                // into the first 32 columns of that half's 64
                mma_ts(tmem + Cfg::kO, tmem + Cfg::kS + 128 * sb + 64 * (kk / 4) + 8 * (kk % 4),
                       desc_join(vb + kk * ((16 * 128) >> 4), dhi), idPV, i > 0 || kk > 0);
              mma_commit(&pv_done[sb]);
              mma_commit(&v_empty[sl]);
              if (i == nt - 1) mma_commit(o_final);
            }
          }
          g += nt;
          ++un;
        }
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
    // -------------------------------------------------------- softmax ---
    // Two warps per TMEM lane quadrant: warps w and w + 4 read the same 32 rows
    // and split every row's columns in half.  The halves agree on the row max
    // through a shared-memory exchange each tile and add their row sums at the
    // end, so both apply identical scaling to their columns.
    const int quad = warp & 3, hf = warp >> 2;
    const int r = quad * 32 + lane;        // query row within the tile = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    constexpr int kHalfS = kBN / 2;        // S columns per half
    constexpr int kHalfD = D / 2;          // O columns per half
    const uint32_t tO = tmem + lane_base + Cfg::kO + hf * kHalfD;
    const float sl2 = a.scale_log2;
    constexpr float kLn2 = 0.6931471805599453f;
    constexpr float kLog2e = 1.4426950408889634f;
    int g = 0, un = 0, xc = 0;
    bool ok = true;
    RowState prev{};
    bool have_prev = false;

    // The two warps of a quadrant meet at named barrier 1 + quad.  Once the CTA
    // is aborting nobody enters it any more, and a warp that leaves the unit
    // loop early arrives there once on its way out, so a partner already
    // waiting is released: the barrier never waits for a warp that has gone.
    auto pair_sync = [&]() -> bool {
      if (__any_sync(0xffffffffu, *abort != 0)) return false;
      named_barrier(1 + quad, 64);
      return true;
    };
    // The partner half's value for this row.  Exchange k writes slot k & 1; the
    // partner reads it before it reaches exchange k + 1, so the slot is free
    // again by exchange k + 2.
    auto exchange = [&](float v, float& o) -> bool {
      float* slot = xch + (xc & 1) * 256;
      slot[hf * 128 + r] = v;
      if (!pair_sync()) return false;
      o = slot[(hf ^ 1) * 128 + r];
      ++xc;
      return true;
    };

    // normalise (and, in the local pass, merge) this half of O of the finished unit
    auto epilogue = [&](const RowState& s, int unit_index) -> bool {
      float l_other;
      if (!exchange(s.l, l_other)) return false;
      const float l = s.l + l_other;
      if (!warp_wait(o_final, unit_index & 1, abort, a.err, a.wait_ns)) return false;
      tc_fence_after();
      const size_t qrow = static_cast<size_t>(s.zq) * a.n;
      float c1 = l > 0.f ? 1.f / l : 0.f, c2 = 0.f;
      float lse2 = s.m + log2f(l);
      const bool far = MODE == kModeLocal && s.valid && s.far;
      if (far) {
        const float lf2 = s.lse_far * kLog2e;
        const float mm = fmaxf(lse2, lf2);
        const float e1 = ex2f(lse2 - mm), e2 = ex2f(lf2 - mm);
        const float den = e1 + e2;
        c1 = e1 / (l * den);
        c2 = e2 / den;
        lse2 = mm + log2f(den);
      }
      if (is_group_mode(MODE)) {
        // rows are scattered by perm: the tile is staged in shared memory with
        // each row's O_far row index (rows past the item go to the spare rows
        // after the last plane), and the V load warp scatters it with TMA once
        // it has read the previous unit's tile out of the stage
        if (unit_index > 0 && !warp_wait(ost_free, (unit_index - 1) & 1, abort, a.err, a.wait_ns)) return false;
        const bool write = s.valid && l > 0.f;
#pragma unroll
        for (int c0 = 0; c0 < kHalfD; c0 += 32) {
          uint32_t ou[32];
          tmem_ld32(tO + c0, ou);
          tmem_wait_ld();
          if (c0 + 32 == kHalfD) {
            tc_fence_before();
            warp_arrive(o_free, lane);
          }
#pragma unroll
          for (int cc = 0; cc < 32; cc += 8) {
            const int v = (hf * kHalfD + c0 + cc) >> 3;
            uint4 o4;
            o4.x = pack_bf16x2(__uint_as_float(ou[cc + 0]) * c1, __uint_as_float(ou[cc + 1]) * c1);
            o4.y = pack_bf16x2(__uint_as_float(ou[cc + 2]) * c1, __uint_as_float(ou[cc + 3]) * c1);
            o4.z = pack_bf16x2(__uint_as_float(ou[cc + 4]) * c1, __uint_as_float(ou[cc + 5]) * c1);
            o4.w = pack_bf16x2(__uint_as_float(ou[cc + 6]) * c1, __uint_as_float(ou[cc + 7]) * c1);
            *reinterpret_cast<uint4*>(sO + (v >> 3) * Cfg::kChunk + r * 128 + (((v & 7) ^ (r & 7)) << 4)) = o4;
          }
        }
        if (hf == 0) {
          row_tok[r] = s.valid ? s.zq * a.m + s.pos : a.B * a.H * a.m + r;
          if (write) a.lse_far[static_cast<size_t>(s.zq) * a.m + s.pos] = lse2 * kLn2;
        }
        fence_proxy_async_smem();
        warp_arrive(ost_full, lane);
        return true;
      }
      // local and dense: the tile goes through the shared-memory stage (same
      // 128 B-swizzled layout as the TMA boxes) and leaves with one TMA store;
      // in the local pass the stage already holds the group partial of the
      // rows.  The stage is free once the V load warp has stored the previous
      // unit's tile out of it: in the local pass that is implied by the group
      // partial it loads there afterwards; in the dense pass it is signalled.
      if (MODE == kModeLocal && !warp_wait(ofar_full, unit_index & 1, abort, a.err, a.wait_ns)) return false;
      if (MODE == kModeDense && unit_index > 0 &&
          !warp_wait(ost_free, (unit_index - 1) & 1, abort, a.err, a.wait_ns))
        return false;
#pragma unroll
      for (int c0 = 0; c0 < kHalfD; c0 += 32) {
        uint32_t ou[32];
        tmem_ld32(tO + c0, ou);
        tmem_wait_ld();
        if (c0 + 32 == kHalfD) {
          tc_fence_before();
          warp_arrive(o_free, lane);
        }
#pragma unroll
        for (int cc = 0; cc < 32; cc += 8) {
          const int v = (hf * kHalfD + c0 + cc) >> 3;
          uint4* slot = reinterpret_cast<uint4*>(sO + (v >> 3) * Cfg::kChunk + r * 128 + (((v & 7) ^ (r & 7)) << 4));
          float f[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(ou[cc + e]) * c1;
          if (far) {
            const uint4 g4 = *slot;
            const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&g4);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 gv = __bfloat1622float2(g2[e]);
              f[2 * e] = fmaf(gv.x, c2, f[2 * e]);
              f[2 * e + 1] = fmaf(gv.y, c2, f[2 * e + 1]);
            }
          }
          uint4 o4;
          o4.x = pack_bf16x2(f[0], f[1]);
          o4.y = pack_bf16x2(f[2], f[3]);
          o4.z = pack_bf16x2(f[4], f[5]);
          o4.w = pack_bf16x2(f[6], f[7]);
          *slot = o4;
        }
      }
      // the tile is in the stage (and visible to the async proxy) once all
      // eight warps have arrived; the V load warp stores it
      fence_proxy_async_smem();
      warp_arrive(ost_full, lane);
      if (hf == 0 && s.valid && a.lse) a.lse[qrow + s.pos] = lse2 * kLn2;
      return true;
    };

    UnitWalk<MODE> walk;
    walk.begin(a, n_units);
    for (int k = 0; ok; ++k) {
      Unit U;
      const int u = walk.step(a, k, U);
      if (u == -1) break;
      if (u < 0) continue;
      // 1. this unit's rows: their loads are issued before the previous
      // unit's epilogue, which hides their latency
      RowState st{};
      st.valid = r < U.nrows;
      st.prob = U.prob;
      st.zq = U.zq;
      st.row0 = U.row0;
      st.far = false;
      int lo = 1, hi = 0;
      st.pos = -1;
      // split index: the row's and the unit's last row's far prefix in every
      // sub-run, loaded here with the rest of the row state so the tile loop
      // never waits on them
      int rowb[kMaxSub], lastb[kMaxSub];
      if (MODE == kModeGroupSplit) {
        const int32_t* lf = a.farlen_sub + (static_cast<size_t>(U.prob) * a.m + U.row0 + U.nrows - 1) * a.nsub;
        const int32_t* rf = a.farlen_sub + (static_cast<size_t>(U.prob) * a.m + U.row0 + min(r, U.nrows - 1)) * a.nsub;
#pragma unroll
        for (int q = 0; q < kMaxSub; ++q) {
          lastb[q] = q < a.nsub ? lf[q] : 0;
          rowb[q] = q < a.nsub && st.valid ? rf[q] : 0;
        }
      }
      if (is_group_mode(MODE)) {
        if (st.valid) {
          const size_t sidx = static_cast<size_t>(U.prob) * a.m + U.row0 + r;
          st.pos = a.perm[sidx];       // the row's item: O_far row within the head
          lo = 0;
          // split top-2 index: the row's far prefix per key sub-run, read as
          // the tile loop enters each sub-run
          if (MODE == kModeGroup) hi = (a.farlen_sub ? a.farlen_sub[sidx * a.nsub + U.sub] : a.farlen_slot[sidx]) - 1;
        }
      } else if (st.valid) {
        st.pos = U.row0 + r;
        lo = st.pos - a.w + 1;
        hi = st.pos;
        if (MODE == kModeLocal) {
          // this row's group partial: flag and LSE now, O row into L2
          st.far = a.farlen_tok[static_cast<size_t>(U.prob) * a.n + st.pos] > 0;
          if (st.far) {
            const size_t qi = static_cast<size_t>(U.zq) * a.n + st.pos;
            st.lse_far = a.lse_far[qi];
            const char* row = reinterpret_cast<const char*>(static_cast<const __nv_bfloat16*>(a.O_far) + qi * D);
            asm volatile("prefetch.global.L2 [%0];" ::"l"(row + hf * D));
          }
        }
      }
      // 2. the previous unit's epilogue overlaps this unit's first S products
      if (have_prev) {
        if (!epilogue(prev, un - 1)) { ok = false; break; }
        have_prev = false;
      }
      // 3. this unit's key tiles
      float m_run = -INFINITY, l = 0.f;
      const int nt = U.t1 - U.t0 + 1;
      // split index: current sub-run column, tile within it, and its tiles
      int sj = -1, stt = 0, snt = 0;
      auto next_sub = [&]() {
        for (++sj; sj < a.nsub; ++sj) {
          const int keys = pick(lastb, sj);
          if (keys > 0) {
            snt = (keys + kBN - 1) / kBN;
            stt = 0;
            hi = st.valid ? pick(rowb, sj) - 1 : -1;
            return;
          }
        }
      };
      if (MODE == kModeGroupSplit) next_sub();
      for (int i = 0; i < nt; ++i) {
        const int gg = g + i;
        // first key of this half (split index: within the current sub-run)
        const int j0 = (MODE == kModeGroupSplit ? stt : U.t0 + i) * kBN + hf * kHalfS;
        const int sb = gg % kSBuf;
        const uint32_t tS = tmem + lane_base + Cfg::kS + 128 * sb + hf * kHalfS;
        if (!warp_wait(&s_full[sb], (gg / kSBuf) & 1, abort, a.err, a.wait_ns)) { ok = false; break; }
        tc_fence_after();
        // this half of the S row: two 32-column loads in flight, one wait
        uint32_t su[kHalfS];
        tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(&su[0]));
        tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&su[32]));
        tmem_wait_ld();
        const bool full = j0 >= lo && j0 + kHalfS - 1 <= hi;
        if (!full) {
#pragma unroll
          for (int cc = 0; cc < kHalfS; ++cc)
            if (j0 + cc < lo || j0 + cc > hi) su[cc] = __float_as_uint(-INFINITY);
        }
        // half-row max: eight independent chains of three-input maxima, a
        // tree, then the partner's half
        float m8[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) m8[j] = fmaxf(__uint_as_float(su[j]), __uint_as_float(su[8 + j]));
#pragma unroll
        for (int cc = 16; cc < kHalfS; cc += 16)
#pragma unroll
          for (int j = 0; j < 8; ++j)
            m8[j] = fmax3(m8[j], __uint_as_float(su[cc + j]), __uint_as_float(su[cc + 8 + j]));
        const float mh = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
        float mo;
        if (!exchange(mh, mo)) { ok = false; break; }
        const float mt = fmaxf(mh, mo);
        const float m_new = fmaxf(m_run, mt * sl2);
        const bool need = m_run != -INFINITY && m_new > m_run + kRescaleThreshold;
        if (m_run == -INFINITY) m_run = m_new;      // nothing accumulated yet for this row
        // O may be rescaled once PV(gg-1) is done.  pv_done[b] completes one
        // phase per PV from buffer b (gg = b, b + kSBuf, ...); S(gg-1), which
        // this thread has read, was issued after PV(gg-1-kSBuf), so the
        // barrier of buffer (gg-1) % kSBuf is at most one phase behind.
        const bool pv_prev = i > 0;
        if (pv_prev && __any_sync(0xffffffffu, need)) {
          const int pb = (gg - 1) % kSBuf;
          if (!warp_wait(&pv_done[pb], ((gg - 1) / kSBuf) & 1, abort, a.err, a.wait_ns)) { ok = false; break; }
          tc_fence_after();
          const float alpha = need ? ex2f(m_run - m_new) : 1.f;
          uint32_t rr[32];
#pragma unroll
          for (int cc = 0; cc < kHalfD; cc += 32) {
            tmem_ld32(tO + cc, rr);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * alpha);
            tmem_st32(tO + cc, rr);
          }
          if (need) {
            l *= alpha;
            m_run = m_new;
          }
        }
        const float mu = m_run == -INFINITY ? 0.f : m_run;
        // p = 2^(s*scale*log2e - m): scale-and-shift in packed pairs, exp2 per
        // element, four packed partial sums; P is written as bf16 pairs over
        // the first 32 of this half's 64 S columns, already read above
        const uint64_t sc2 = f2_pack(sl2, sl2), nm2 = f2_pack(-mu, -mu);
        uint64_t acc[4] = {0, 0, 0, 0};
        uint32_t pk[kHalfS / 2];
#pragma unroll
        for (int cc = 0; cc < kHalfS; cc += 2) {
          float t0, t1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(su[cc]), __uint_as_float(su[cc + 1])), sc2, nm2), t0, t1);
          const float p0 = ex2f(t0), p1 = ex2f(t1);
          acc[(cc >> 1) & 3] = f2_add(acc[(cc >> 1) & 3], f2_pack(p0, p1));
          pk[cc / 2] = pack_bf16x2(p0, p1);
        }
        tmem_st32(tS, pk);
        {
          const uint64_t s2 = f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3]));
          float s0, s1;
          f2_unpack(s2, s0, s1);
          l += s0 + s1;
        }
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(&p_ready[sb], lane);
        if (MODE == kModeGroupSplit && ++stt == snt) next_sub();   // the next tile's sub-run
      }
      if (!ok) break;
      g += nt;
      st.m = m_run;
      st.l = l;
      prev = st;
      have_prev = true;
      ++un;
    }
    if (ok && have_prev) ok = epilogue(prev, un - 1);
    if (!ok) named_barrier_arrive(1 + quad, 64);   // release a partner waiting at the pair barrier
  }

  __syncwarp();          // lanes of the load and MMA warps reconverge before the CTA barrier
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpPV) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

// K_s[b, kv, s, :] = K[b, kv, perm_a[s] >> kshift, :] (and V), a = assignment
// of kv; s runs over the m sorted items, K has n rows per head.
__global__ void __launch_bounds__(256) permute_kv_kernel(const uint4* __restrict__ K,
                                                         const uint4* __restrict__ V,
                                                         uint4* __restrict__ Ks,
                                                         uint4* __restrict__ Vs,
                                                         const int32_t* __restrict__ perm, int H_kv,
                                                         int n, int m, int kshift, int vec_per_row,
                                                         int A, long long total) {
  for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = e / vec_per_row;
    const int u = static_cast<int>(e % vec_per_row);
    const int s = static_cast<int>(row % m);
    const long long bk = row / m;             // b * H_kv + kv
    const int kvh = static_cast<int>(bk % H_kv);
    const long long bb = bk / H_kv;
    const long long p = bb * A + (A == 1 ? 0 : kvh);
    const int src = __ldg(perm + p * m + s) >> kshift;
    const long long si = (bk * n + src) * vec_per_row + u;
    Ks[e] = __ldg(K + si);
    Vs[e] = __ldg(V + si);
  }
}

template <int D>
cudaError_t launch_d(const AttnArgs& a, const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                     const CUtensorMap* tm_v, const CUtensorMap* tm_o, const CUtensorMap* tm_of, int mode,
                     int max_items, int num_sms, cudaStream_t st) {
  using Cfg = AttnCfg<D>;
  long long units;
  if (is_group_mode(mode)) {
    const int hpa = a.A == 1 ? a.H : a.H / a.H_kv;
    units = static_cast<long long>(max_items) * hpa;
  } else {
    units = static_cast<long long>(a.B) * a.H * ((a.n + kBM - 1) / kBM);
  }
  if (units == 0) return cudaSuccess;
  const unsigned grid = static_cast<unsigned>(units < num_sms ? units : num_sms);
  if (mode == kModeGroup)
    attn_tc_kernel<D, kModeGroup><<<grid, kThreads, Cfg::kSmem, st>>>(*tm_q, *tm_k, *tm_v, *tm_o, *tm_of, a);
  else if (mode == kModeGroupSplit)
    attn_tc_kernel<D, kModeGroupSplit><<<grid, kThreads, Cfg::kSmem, st>>>(*tm_q, *tm_k, *tm_v, *tm_o, *tm_of, a);
  else if (mode == kModeLocal)
    attn_tc_kernel<D, kModeLocal><<<grid, kThreads, Cfg::kSmem, st>>>(*tm_q, *tm_k, *tm_v, *tm_o, *tm_of, a);
  else
    attn_tc_kernel<D, kModeDense><<<grid, kThreads, Cfg::kSmem, st>>>(*tm_q, *tm_k, *tm_v, *tm_o, *tm_of, a);
  return cudaGetLastError();
}

template <int D>
cudaError_t set_smem() {
  using Cfg = AttnCfg<D>;
  cudaError_t e;
  e = cudaFuncSetAttribute(attn_tc_kernel<D, kModeGroup>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(attn_tc_kernel<D, kModeGroupSplit>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(attn_tc_kernel<D, kModeLocal>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(attn_tc_kernel<D, kModeDense>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
}

}  // namespace

cudaError_t launch_permute_kv_bf16(const void* K, const void* V, void* Ks, void* Vs,
                                   const int32_t* perm, int B, int H_kv, int n, int m, int kshift,
                                   int d, int A, cudaStream_t st) {
  const int vpr = d / 8;
  const long long total = static_cast<long long>(B) * H_kv * m * vpr;
  if (total == 0) return cudaSuccess;
  const long long want = (total + 255) / 256;
  const int grid = static_cast<int>(want < 152LL * 16 ? want : 152LL * 16);
  permute_kv_kernel<<<grid, 256, 0, st>>>(static_cast<const uint4*>(K), static_cast<const uint4*>(V),
                                          static_cast<uint4*>(Ks), static_cast<uint4*>(Vs), perm,
                                          H_kv, n, m, kshift, vpr, A, total);
  return cudaGetLastError();
}

cudaError_t launch_attn_tc_bf16(const AttnArgs& a, const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                const CUtensorMap* tm_v, const CUtensorMap* tm_o, const CUtensorMap* tm_of,
                                int d, int mode, int max_items, int num_sms, cudaStream_t st) {
  if (d == 64) return launch_d<64>(a, tm_q, tm_k, tm_v, tm_o, tm_of, mode, max_items, num_sms, st);
  if (d == 128) return launch_d<128>(a, tm_q, tm_k, tm_v, tm_o, tm_of, mode, max_items, num_sms, st);
  return cudaErrorInvalidValue;
}

cudaError_t setup_attn_kernels() {
  cudaError_t e = set_smem<64>();
  if (e != cudaSuccess) return e;
  return set_smem<128>();
}

}  // namespace focus
