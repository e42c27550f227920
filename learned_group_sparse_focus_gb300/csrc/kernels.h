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

// Bits of the device error word (first int of the workspace).
enum : int {
  kErrBadGroup = 1,   // a group id outside [0, K)
  kErrTimeout = 2,    // a bounded wait ran out
  kErrInternal = 4,   // an index or item failed a consistency check
};

struct IndexLaunch {
  const int32_t* gid;
  int P, A, n, K, w_eff;
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
  int32_t* gid;    // [B, A, n]
  int B, n, D, d_g, K, A;
  int* err;
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
  float scale_log2;          // scale * log2(e)
  int* err;
};

// index.cu
cudaError_t launch_build_index(const IndexLaunch& L, cudaStream_t st);
cudaError_t setup_index_kernels();

// assign.cu
cudaError_t launch_assign_f32(const AssignLaunch& L, cudaStream_t st);
cudaError_t launch_assign_bf16(const AssignLaunch& L, const CUtensorMap* tm_h,
                               const CUtensorMap* tm_w, cudaStream_t st);
cudaError_t setup_assign_kernels();

// attn_simt.cu (fp32 storage, fp32 arithmetic on the CUDA cores)
enum AttnMode : int { kModeLocal = 0, kModeGroup = 1, kModeDense = 2 };
cudaError_t launch_attn_simt_f32(const AttnArgs& a, int d, int mode, int max_items,
                                 cudaStream_t st);

// attn_tc.cu (bf16 storage, tcgen05 tensor cores, fp32 softmax)
cudaError_t launch_permute_kv_bf16(const void* K, const void* V, void* Ks, void* Vs,
                                   const int32_t* perm, int B, int H_kv, int n, int d, int A,
                                   cudaStream_t st);
// tm_o / tm_of: O and the group partial O_far as {d, n, B*H} tiles (local and
// dense passes store O, and the local pass loads O_far, through them).
cudaError_t launch_attn_tc_bf16(const AttnArgs& a, const CUtensorMap* tm_q,
                                const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                const CUtensorMap* tm_o, const CUtensorMap* tm_of, int d, int mode,
                                int max_items, int num_sms, cudaStream_t st);
cudaError_t setup_attn_kernels();

}  // namespace focus
