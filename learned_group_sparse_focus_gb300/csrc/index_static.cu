// focus_build_index_static: the group-sorted index built with no workspace
// and no allocation of any kind.
//
// Some callers cannot allocate device memory at the point where they need the
// index: a serving loop that fixes its memory footprint at start-up and must
// not grow it (or pay the device-wide synchronisation that cudaMalloc and
// cudaFree can cause) while requests are in flight, and callers that only want
// the index, for whom the regular workspace (sized for the attention pass's
// permuted K/V and partial outputs) is gigabytes of memory they do not have.
// Such a caller owns its output buffers; the only scratch the sort needs
// (per-segment histograms, tile bases and item costs) lives in one fixed
// file-scope device array below.
//
// The arithmetic is exactly focus_build_index's: the same five launches run
// with the scratch pointers moved, so the outputs are bit-identical.
#include <cstdint>
#include <mutex>

#include "kernels.h"

namespace focus {
namespace {

constexpr size_t kScratchBytes = FOCUS_INDEX_STATIC_SCRATCH_BYTES;
constexpr size_t kScratchAlign = 256;

// Every word of it that a call reads, that call has written first, so nothing
// in it has to start at zero.  Two calls whose kernels overlap in time (other
// streams, other host threads) share it and race; callers must order them.
__device__ __align__(256) int32_t g_index_scratch[kScratchBytes / sizeof(int32_t)];

std::mutex g_static_mu;
bool g_static_ready[64] = {};
int32_t* g_static_ptr[64] = {};

size_t round_up(size_t x) { return (x + kScratchAlign - 1) & ~(kScratchAlign - 1); }

bool aligned(const void* p, uintptr_t a) { return p && (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Device address of g_index_scratch for the current device, looked up once per
// device (with that device current); also raises the index kernels' shared
// memory limit there.
focus_status_t static_setup(int32_t** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FOCUS_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (!g_static_ready[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_index_scratch) != cudaSuccess || !ptr) return FOCUS_ERR_CUDA;
    if (setup_index_kernels() != cudaSuccess) return FOCUS_ERR_CUDA;
    g_static_ptr[dev] = static_cast<int32_t*>(ptr);
    g_static_ready[dev] = true;
  }
  *out = g_static_ptr[dev];
  return FOCUS_OK;
}

}  // namespace
}  // namespace focus

using namespace focus;

extern "C" {

focus_status_t focus_build_index_static(const focus_params_t* p, const int32_t* gid,
                                        focus_index_t* idx, int32_t* err, void* stream) {
  // the same problems focus_build_index accepts
  if (!p || focus_workspace_bytes(p) == 0) return FOCUS_ERR_INVALID_ARG;
  if (!idx || !aligned(gid, 16) || !aligned(err, kScratchAlign)) return FOCUS_ERR_INVALID_ARG;
  if (!aligned(idx->counts, 16) || !aligned(idx->offsets, 16) || !aligned(idx->perm, 16) ||
      !aligned(idx->rank, 16) || !aligned(idx->farlen_tok, 16) || !aligned(idx->farlen_slot, 16) ||
      !aligned(idx->items, 16) || !aligned(idx->order, 16) || !aligned(idx->n_items, 16))
    return FOCUS_ERR_INVALID_ARG;
  const size_t P = static_cast<size_t>(p->B) * p->A;
  const size_t n = static_cast<size_t>(p->n), K = static_cast<size_t>(p->K);
  const size_t nseg = (n + kIndexSeg - 1) / kIndexSeg;
  const size_t max_items = P * ((n + kTileM - 1) / kTileM + (K < n ? K : n));
  if (idx->max_items < 0 || static_cast<size_t>(idx->max_items) < max_items) return FOCUS_ERR_INVALID_ARG;

  // scratch carve-up: histograms, tile bases, item costs
  const size_t o_seg = 0;
  const size_t o_tb = round_up(o_seg + P * nseg * K * sizeof(int32_t));
  const size_t o_cost = round_up(o_tb + P * (K + 1) * sizeof(int32_t));
  const size_t need = round_up(o_cost + max_items * sizeof(int32_t));
  if (need > kScratchBytes) return FOCUS_ERR_WORKSPACE;

  int32_t* base = nullptr;
  if (focus_status_t s = static_setup(&base)) return s;
  char* b = reinterpret_cast<char*>(base);

  IndexLaunch il{};
  il.gid = gid;
  il.P = static_cast<int>(P);
  il.A = p->A;
  il.n = p->n;
  il.K = p->K;
  il.w_eff = p->w > 1 ? p->w : 1;
  il.segcnt = reinterpret_cast<int32_t*>(b + o_seg);
  il.counts = idx->counts;
  il.offsets = idx->offsets;
  il.tile_base = reinterpret_cast<int32_t*>(b + o_tb);
  il.perm = idx->perm;
  il.rank = idx->rank;
  il.farlen_tok = idx->farlen_tok;
  il.farlen_slot = idx->farlen_slot;
  il.items = idx->items;
  il.cost = reinterpret_cast<int32_t*>(b + o_cost);
  il.order = idx->order;
  il.n_items = idx->n_items;
  il.max_items = static_cast<int>(max_items);
  il.err = err;
  if (launch_build_index(il, static_cast<cudaStream_t>(stream)) != cudaSuccess) return FOCUS_ERR_CUDA;
  idx->max_items = static_cast<int32_t>(max_items);
  idx->w_eff = il.w_eff;
  return FOCUS_OK;
}

}  // extern "C"
