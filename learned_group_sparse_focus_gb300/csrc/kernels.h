// Launch descriptions shared by the host ABI layer and the kernel files.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/focus.h"

namespace focus {

constexpr int kTileM = FOCUS_TILE_M;   // query rows per group-pass work item
constexpr int kTileN = FOCUS_TILE_N;   // keys per attention tile
constexpr int kMaxK = FOCUS_MAX_K;
constexpr int kIndexSeg = 1024;        // tokens per counting-sort segment
// One second: no wait in these kernels legitimately lasts this long.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

// Bits of the device error word (first int of the workspace).
enum : int {
  kErrBadGroup = 1,   // a group id outside [0, K)
  kErrTimeout = 2,    // a bounded wait ran out
  kErrInternal = 4,   // an index or item failed a consistency check
};

// n counts the sorted items: tokens, or for top-k membership the n_tok * k
// entries (entry e = i * k + c, token i = e >> kshift); positions compared
// against the window are token positions.
struct IndexLaunch {
  const int32_t* gid;
  int P, A, n, K, w_eff;
  int kshift;           // 0: items are tokens; log2(k): items are entries
  int32_t* segcnt;      // [P][nseg][K]
  int32_t* counts;      // [P][K]
  int32_t* offsets;     // [P][K+1]
  int32_t* tile_base;   // [P][K+1]
  int32_t* perm;        // [P][n]
  int32_t* rank;        // [P][n]
  int32_t* farlen_tok;  // [P][n]
  int32_t* farlen_slot; // [P][n]
  focus_item_t* items;  // [max_items]
  int32_t* cost;        // [max_items]
  int32_t* order;       // [max_items]
  int32_t* n_items;     // [1]
  int max_items;
  int* err;
};

struct AssignLaunch {
  const void* h;   // [B*n, D]
  const void* W;   // [A*d_g, D]
  const void* C;   // [A, K, d_g]
  int32_t* gid;    // [B, A, n, topk]
  int B, n, D, d_g, K, A;
  int topk;        // 1 or 2 ids per token, best first
  int* err;
  float* scores;   // non-null: write every score [B, A, n, K] (fp32) instead of ids
  int num_sms;     // SMs of the device (persistent grid)
  int tile_rows;   // tokens per tile = rows of tm_h's box (assign_tile_rows)
};

// Everything the attention kernels read besides the K/V tensor maps.
struct AttnArgs {
  const void* Q;             // [B, H, n, d]
  void* O;                   // [B, H, n, d]   final output (local / dense pass)
  float* lse;                // [B, H, n] or null
  void* O_far;               // [B, H, n, d]   group-pass partial, normalised
  float* lse_far;            // [B, H, n]      group-pass partial LSE (natural log)
  const void* Kg;            // [B, H_kv, n, d] keys for the SIMT path (natural order)
  const void* Vg;            // [B, H_kv, n, d]
  const int32_t* perm;       // [B*A][n]
  const int32_t* farlen_tok; // [B*A][n]
  const int32_t* farlen_slot;// [B*A][n]
  const focus_item_t* items;
  const int32_t* order;
  const int32_t* n_items;
  int B, H, H_kv, n, A, w;   // w: effective window (>= 1)
  // group pass only: sorted items per problem (perm, farlen_slot and the
  // O_far / lse_far rows are indexed by item) and the item -> token shift.
  // m = n, kshift = 0 for one group per token; m = n * k for top-k entries.
  int m, kshift;
  float scale_log2;          // scale * log2(e)
  int* err;
  // Bounded waits give up after wait_ns.  Test hook: with hold_first_q set the
  // Q load warp never issues its first Q tile, so the first S product's wait
  // runs out and the kernel takes its abort path.
  unsigned long long wait_ns;
  int hold_first_q;
  // group pass over a top-2 split index: per-row bounds from farlen_sub
  // [m][nsub] (column = the item's pad) instead of farlen_slot; else null
  const int32_t* farlen_sub;
  int nsub;
  const int32_t* offsets;    // split index: [B*A][K*K + 1] sub-run starts
};

// index.cu
cudaError_t launch_build_index(const IndexLaunch& L, cudaStream_t st);
// Top-2 split index: L describes the 2n entries with their virtual group
// ids v = g * K + o (L.gid, L.K = K * K, L.kshift = 1); farlen_sub
// [P][2n][K - 1] receives each slot's far prefix in every sub-run (g, o') of its
// group, L.farlen_tok / L.farlen_slot the entry's / slot's total, and the work
// list holds one item per (row tile, sub-run) with item.pad = the sub-run's
// column.  Each far pair is visited once: in the pass of the smaller group the
// two tokens share.
cudaError_t launch_build_index_split(const IndexLaunch& L, int K, int32_t* farlen_sub, cudaStream_t st);
cudaError_t setup_index_kernels();

// assign.cu
cudaError_t launch_assign_f32(const AssignLaunch& L, cudaStream_t st);
cudaError_t launch_assign_bf16(const AssignLaunch& L, const CUtensorMap* tm_h,
                               const CUtensorMap* tm_w, cudaStream_t st);
cudaError_t setup_assign_kernels();
// Tokens per tile of the bf16 assign kernel for `tokens` tokens and ncol = A * d_g
// projection columns: 128, or (persistent kernel, more than one tile per SM) the
// smallest count that gives every SM the same number of tiles.
int assign_tile_rows(int tokens, int ncol, int num_sms);

// attn_simt.cu (fp32 storage, fp32 arithmetic on the CUDA cores)
// kModeGroupSplit: the group pass over a split top-2 index (each unit walks
// its row tile's key sub-runs one after another; see launch_build_index_split)
enum AttnMode : int { kModeLocal = 0, kModeGroup = 1, kModeDense = 2, kModeGroupSplit = 3 };
__host__ __device__ constexpr bool is_group_mode(int mode) { return mode == kModeGroup || mode == kModeGroupSplit; }
cudaError_t launch_attn_simt_f32(const AttnArgs& a, int d, int mode, int max_items,
                                 cudaStream_t st);

// attn_tc.cu (bf16 storage, tcgen05 tensor cores, fp32 softmax)
// Ks[b, kv, s] = K[b, kv, perm[s] >> kshift] for the m sorted items s of kv's
// assignment (and V); K/V have n rows per head, Ks/Vs have m.
cudaError_t launch_permute_kv_bf16(const void* K, const void* V, void* Ks, void* Vs,
                                   const int32_t* perm, int B, int H_kv, int n, int m, int kshift,
                                   int d, int A, cudaStream_t st);
// tm_o / tm_of: O and the group partial O_far as {d, n, B*H} tiles (local and
// dense passes store O, and the local pass loads O_far, through them).
cudaError_t launch_attn_tc_bf16(const AttnArgs& a, const CUtensorMap* tm_q,
                                const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                const CUtensorMap* tm_o, const CUtensorMap* tm_of, int d, int mode,
                                int max_items, int num_sms, cudaStream_t st);
cudaError_t setup_attn_kernels();

// topk.cu (top-2 membership)
// vg[p, 2i + c] = g_c * K + g_(1-c) for token i's groups g_0, g_1 (the split
// index's virtual group ids); equal or out-of-range ids raise kErrBadGroup.
cudaError_t launch_split_ids(const int32_t* gid2, int P, int n, int K, int32_t* vg, int* err, cudaStream_t st);
// pair_gid[p, i] = id of token i's two groups {a, b} (a < b) among the
// K (K - 1) / 2 pairs; equal or out-of-range ids raise kErrBadGroup.
cudaError_t launch_pair_ids(const int32_t* gid2, int P, int n, int K, int32_t* pair_gid, int* err,
                            cudaStream_t st);
// far_any[p, i] = 1 if either entry of token i has far keys, else 0.
cudaError_t launch_far_any(const int32_t* farlen_entry, int P, int n, int32_t* far_any,
                           cudaStream_t st);
// Per query row: the two entry partials minus the pair partial, combined by
// log-sum-exp into one far partial per token (O_far, lse_far).
struct MergeLaunch {
  const void* O_e;              // [B*H*2n (+ spare), d]  entry partials
  const float* lse_e;           // [B*H*2n]
  const void* O_p;              // [B*H*n (+ spare), d]   pair partials
  const float* lse_p;           // [B*H*n]
  const int32_t* farlen_entry;  // [B*A][2n]
  const int32_t* farlen_pair;   // [B*A][n]
  void* O_far;                  // [B*H*n (+ spare), d]
  float* lse_far;               // [B*H*n]
  int B, H, H_kv, A, n, d;
};
cudaError_t launch_topk_merge(const MergeLaunch& L, int dtype, cudaStream_t st);

// two_call.cu: the two-call comparator's separate log-sum-exp combine of the
// window call's output (in place in O) with the group partial.
struct CombineLaunch {
  void* O;                      // [B*H*n, d] in: window-call output, out: merged
  const float* lse_loc;         // [B*H*n]    window-call LSE
  const void* O_far;            // [B*H*n (+ spare), d] group partial
  const float* lse_far;         // [B*H*n]
  const int32_t* farlen_tok;    // [B*A][n]   > 0: the row has far keys
  float* lse_out;               // [B*H*n] merged LSE, or null (must not alias lse_loc)
  int B, H, H_kv, A, n, d;
};
cudaError_t launch_lse_combine(const CombineLaunch& L, int dtype, cudaStream_t st);

// sinkhorn.cu: Sinkhorn soft assignment over S [P, n, K] (fp32).
struct SinkhornLaunch {
  const float* S;    // [P, n, K] scores
  float* G;          // [P, n, K] output (may alias S)
  float* u;          // [P, n] row potentials
  float* v;          // [P, K] column potentials
  float2* part;      // [P, chunks, K] per-chunk column (max, sum)
  int* ticket;       // [P] blocks of the current pass done (0 between launches)
  int P, n, K;
  float inv_tau;
  int* err;          // device error word (bounded waits)
  int num_sms;
};
int sinkhorn_rows_per_chunk(int n);
cudaError_t setup_sinkhorn_kernels();

// attn_bwd.cu: backward over the kept pairs (fp32 arithmetic on the CUDA cores).
struct BwdArgs {
  const void *Q, *K, *V, *O, *dO;   // forward tensors and the upstream gradient
  const float* lse;                 // [B, H, n] forward LSE (natural log)
  float* delta;                     // [B, H, n] dO . O
  float* dq_far;                    // [B*H*n, d]    far-key part of dQ
  float *dk_far, *dv_far;           // [B*H_kv*n, d] far-query parts of dK, dV
  void *dQ, *dK, *dV;               // outputs (dtype of Q)
  const int32_t *perm, *farlen_tok, *farlen_slot, *offsets;
  const focus_item_t* items;
  const int32_t* order;
  const int32_t* n_items;
  int B, H, H_kv, n, d, A, groups, w;   // groups: K, the number of centroids
  float scale, scale_log2;
  int* err;                         // device error word (bounded waits)
  const float *lse_sorted, *delta_sorted;  // bf16 path: LSE and Delta in each head's index order
  int* ticket;                      // bf16 path: unit counter of the far dK/dV kernel, zero at launch
  int32_t* kv_order;                // bf16 path: far dK/dV units, longest first [B * H_kv * ceil(n / 128)]
};
cudaError_t launch_attn_bwd(const BwdArgs& a, int dtype, int max_items, cudaStream_t st);
cudaError_t launch_bwd_delta(const BwdArgs& a, int dtype, cudaStream_t st);

// attn_bwd_tc.cu: the same backward for bf16 on the tcgen05 tensor cores (after
// launch_bwd_delta and the index-order copies).  All maps {d, n, planes} with
// 128-row boxes: *s over the index-ordered copies (group kernels), *3 over the
// inputs (window kernels).
cudaError_t launch_attn_bwd_tc(const BwdArgs& a, const CUtensorMap* qs, const CUtensorMap* dos,
                               const CUtensorMap* ks, const CUtensorMap* vs, const CUtensorMap* q3,
                               const CUtensorMap* do3, const CUtensorMap* k3, const CUtensorMap* v3,
                               int max_items, int num_sms, cudaStream_t st);
cudaError_t setup_bwd_tc_kernels();
// Q, dO rows and LSE of every query head sorted by its assignment's index (for
// the group kernels' tile loads), and Delta = rowsum(dO * O) in natural and
// index order.
cudaError_t launch_bwd_permute_q(const BwdArgs& a, void* Qs, void* dOs, float* lse_s, float* delta_s,
                                 cudaStream_t st);
cudaError_t launch_sinkhorn(const SinkhornLaunch& L, int iters, cudaStream_t st);

}  // namespace focus
