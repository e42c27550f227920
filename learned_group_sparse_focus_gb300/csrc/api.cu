// Host side of the Focus C ABI: argument checks, workspace layout, TMA
// descriptors and the launch sequence of each call.  See include/focus.h for
// the contract of every entry point.
#include <cmath>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "kernels.h"

namespace focus {
namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t elt_size(int dtype) { return dtype == FOCUS_BF16 ? 2 : 4; }

// Byte offsets of every region inside the workspace.
struct Layout {
  size_t err, segcnt, counts, offsets, tile_base, perm, rank, far_tok, far_slot, items, cost,
      order, n_items, Ks, Vs, O_far, lse_far, lse_loc, total;
  int nseg, max_items;
};

bool params_ok(const focus_params_t* p) {
  if (!p) return false;
  if (p->B < 1 || p->H < 1 || p->H_kv < 1 || p->H % p->H_kv != 0) return false;
  if (p->n < 1 || p->n > FOCUS_MAX_N) return false;
  if (p->d < 1 || p->D < 1 || p->d_g < 1) return false;
  if (p->K < 1 || p->K > FOCUS_MAX_K) return false;
  if (!(p->A == 1 || p->A == p->H_kv)) return false;
  if (p->w < 0) return false;
  if (!(std::isfinite(p->scale) && p->scale > 0.f)) return false;
  if (p->dtype != FOCUS_F32 && p->dtype != FOCUS_BF16) return false;
  if (static_cast<long long>(p->B) * p->A > 4096) return false;
  return true;
}

Layout layout_of(const focus_params_t* p) {
  Layout L{};
  const size_t P = static_cast<size_t>(p->B) * p->A;
  const size_t n = p->n, K = p->K;
  L.nseg = static_cast<int>((n + kIndexSeg - 1) / kIndexSeg);
  L.max_items = static_cast<int>(P * ((n + kTileM - 1) / kTileM + (K < n ? K : n)));
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align_up(o + bytes);
    return at;
  };
  L.err = take(kAlign);
  L.segcnt = take(P * L.nseg * K * 4);
  L.counts = take(P * K * 4);
  L.offsets = take(P * (K + 1) * 4);
  L.tile_base = take(P * (K + 1) * 4);
  L.perm = take(P * n * 4);
  L.rank = take(P * n * 4);
  L.far_tok = take(P * n * 4);
  L.far_slot = take(P * n * 4);
  L.items = take(static_cast<size_t>(L.max_items) * sizeof(focus_item_t));
  L.cost = take(static_cast<size_t>(L.max_items) * 4);
  L.order = take(static_cast<size_t>(L.max_items) * 4);
  L.n_items = take(4);
  const size_t es = elt_size(p->dtype);
  const size_t kvb = static_cast<size_t>(p->B) * p->H_kv * n * p->d * es;
  L.Ks = take(p->dtype == FOCUS_BF16 ? kvb : 0);
  L.Vs = take(p->dtype == FOCUS_BF16 ? kvb : 0);
  // + one tile of rows that the group pass's row scatter sends rows past an
  // item's end to (never read)
  L.O_far = take((static_cast<size_t>(p->B) * p->H * n + kTileM) * p->d * es);
  L.lse_far = take(static_cast<size_t>(p->B) * p->H * n * 4);
  // the two-call comparator's window-call LSE
  L.lse_loc = take(static_cast<size_t>(p->B) * p->H * n * 4);
  L.total = o;
  return L;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

// ----------------------------------------------------- per-device set-up ---
std::mutex g_mu;
bool g_ready[64] = {};
int g_sms[64] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

focus_status_t ensure_setup() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FOCUS_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return FOCUS_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  if (!g_ready[dev]) {
    if (cudaDeviceGetAttribute(&g_sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        g_sms[dev] < 1)
      return FOCUS_ERR_CUDA;
    if (setup_index_kernels() != cudaSuccess) return FOCUS_ERR_CUDA;
    if (setup_assign_kernels() != cudaSuccess) return FOCUS_ERR_CUDA;
    if (setup_attn_kernels() != cudaSuccess) return FOCUS_ERR_CUDA;
    if (setup_bwd_tc_kernels() != cudaSuccess) return FOCUS_ERR_CUDA;
    if (setup_sinkhorn_kernels() != cudaSuccess) return FOCUS_ERR_CUDA;
    g_ready[dev] = true;
  }
  return FOCUS_OK;
}

// bf16 tensor map over rows of `inner` elements: dims {inner, rows[, planes]}
// (rank 2 or 3, matching the TMA instruction that reads it), box
// {64, box_rows[, 1]}, 128-byte swizzle, zero fill out of bounds.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t planes,
              uint32_t box_rows, int rank) {
  cuuint64_t dims[3] = {inner, rows, planes};
  cuuint64_t strides[2] = {inner * 2, inner * rows * 2};
  cuuint32_t box[3] = {64, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank,
                              const_cast<void*>(base), dims, strides, box, es,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

focus_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? FOCUS_OK : FOCUS_ERR_CUDA; }

// SMs of the current device (valid after ensure_setup).
int sm_count() {
  int dev = 0;
  cudaGetDevice(&dev);
  return (dev >= 0 && dev < 64 && g_sms[dev] > 0) ? g_sms[dev] : 1;
}

focus_status_t check_ws(const focus_params_t* p, void* ws, size_t ws_bytes) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1))) return FOCUS_ERR_INVALID_ARG;
  if (ws_bytes < layout_of(p).total) return FOCUS_ERR_WORKSPACE;
  return FOCUS_OK;
}

AttnArgs attn_args(const focus_params_t* p, const void* Q, const void* K, const void* V, void* O,
                   float* lse, void* ws, const Layout& L) {
  AttnArgs a{};
  a.Q = Q;
  a.O = O;
  a.lse = lse;
  a.O_far = at<void>(ws, L.O_far);
  a.lse_far = at<float>(ws, L.lse_far);
  a.Kg = K;
  a.Vg = V;
  a.B = p->B;
  a.H = p->H;
  a.H_kv = p->H_kv;
  a.n = p->n;
  a.A = p->A;
  a.w = p->w > 1 ? p->w : 1;
  a.m = p->n;
  a.kshift = 0;
  a.scale_log2 = p->scale * 1.4426950408889634f;
  a.err = at<int>(ws, L.err);
  a.wait_ns = kWaitLimitNs;
  a.hold_first_q = 0;
  return a;
}

// ----------------------------------------------- top-k workspace layout ---
// One index (regions of a counting sort over m items into K groups).
struct IndexRegions {
  size_t segcnt, counts, offsets, tile_base, perm, rank, far_tok, far_slot, items, cost, order,
      n_items;
  int nseg, max_items;
};

struct LayoutTopk {
  size_t err, pair_gid, far_any, Ks, Vs, O_e, lse_e, O_p, lse_p, O_far, lse_far, total;
  size_t vgid, far_sub;   // split index: virtual group ids, far prefix per (slot, sub-run)
  IndexRegions ent, pair;
  int k, m, Kp;
  bool split;
};

int pair_count(int K) { return K * (K - 1) / 2; }

// Top-2 with few groups and bf16 tensors uses the split index (memberships
// sorted by (group, other group, position)): it visits every far pair once,
// where the entry and pair indices visit pairs that share both groups twice
// and subtract them once.  A row tile walks the K - 1 sub-runs of its group,
// so the split pays for small K, where shared pairs are common (1 in 6 at
// K = 4).  The fp32 path keeps the entry and pair indices.
constexpr int kSplitMaxK = 8;
bool split_topk(const focus_params_t* p, int k) {
  return k == 2 && p->K <= kSplitMaxK && p->dtype == FOCUS_BF16;
}

bool topk_ok(const focus_params_t* p, int k) {
  if (!params_ok(p) || !(k == 1 || k == 2)) return false;
  if (k == 2 && (p->K < 2 || pair_count(p->K) > FOCUS_MAX_K)) return false;
  return true;
}

LayoutTopk layout_topk(const focus_params_t* p, int k) {
  LayoutTopk L{};
  const size_t P = static_cast<size_t>(p->B) * p->A;
  const size_t n = p->n;
  L.k = k;
  L.m = p->n * k;
  L.split = split_topk(p, k);
  L.Kp = k == 2 && !L.split ? pair_count(p->K) : 0;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align_up(o + bytes);
    return at;
  };
  // mult: work items per row tile (the split index: one per key sub-run)
  auto take_index = [&](IndexRegions& R, size_t m, size_t K, size_t mult) {
    R.nseg = static_cast<int>((m + kIndexSeg - 1) / kIndexSeg);
    R.max_items = static_cast<int>(P * ((m + kTileM - 1) / kTileM + (K < m ? K : m)) * mult);
    R.segcnt = take(P * R.nseg * K * 4);
    R.counts = take(P * K * 4);
    R.offsets = take(P * (K + 1) * 4);
    R.tile_base = take(P * (K + 1) * 4);
    R.perm = take(P * m * 4);
    R.rank = take(P * m * 4);
    R.far_tok = take(P * m * 4);
    R.far_slot = take(P * m * 4);
    R.items = take(static_cast<size_t>(R.max_items) * sizeof(focus_item_t));
    R.cost = take(static_cast<size_t>(R.max_items) * 4);
    R.order = take(static_cast<size_t>(R.max_items) * 4);
    R.n_items = take(4);
  };
  L.err = take(kAlign);
  if (L.split) {
    const size_t K = p->K;
    take_index(L.ent, static_cast<size_t>(L.m), K * K, 1);
    L.vgid = take(P * L.m * 4);
    L.far_sub = take(P * L.m * (K - 1) * 4);
    L.far_any = take(P * n * 4);
  } else {
    take_index(L.ent, static_cast<size_t>(L.m), p->K, 1);
    if (k == 2) {
      take_index(L.pair, n, L.Kp, 1);
      L.pair_gid = take(P * n * 4);
      L.far_any = take(P * n * 4);
    }
  }
  const size_t es = elt_size(p->dtype);
  const size_t qplanes = static_cast<size_t>(p->B) * p->H;
  const size_t kvb = static_cast<size_t>(p->B) * p->H_kv * L.m * p->d * es;
  L.Ks = take(p->dtype == FOCUS_BF16 ? kvb : 0);
  L.Vs = take(p->dtype == FOCUS_BF16 ? kvb : 0);
  if (k == 2) {
    // entry and pair partials, each with the spare tile of rows the row
    // scatter sends rows past an item's end to
    L.O_e = take((qplanes * L.m + kTileM) * p->d * es);
    L.lse_e = take(qplanes * L.m * 4);
    if (!L.split) {
      L.O_p = take((qplanes * n + kTileM) * p->d * es);
      L.lse_p = take(qplanes * n * 4);
    }
  }
  L.O_far = take((qplanes * n + kTileM) * p->d * es);
  L.lse_far = take(qplanes * n * 4);
  L.total = o;
  return L;
}

focus_status_t check_ws_topk(const focus_params_t* p, int k, void* ws, size_t ws_bytes) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1))) return FOCUS_ERR_INVALID_ARG;
  if (ws_bytes < layout_topk(p, k).total) return FOCUS_ERR_WORKSPACE;
  return FOCUS_OK;
}

IndexLaunch index_launch(void* ws, const IndexRegions& R, const int32_t* gid, int P, int A, int n,
                         int K, int w_eff, int kshift, int* err) {
  IndexLaunch il{};
  il.gid = gid;
  il.P = P;
  il.A = A;
  il.n = n;
  il.K = K;
  il.w_eff = w_eff;
  il.kshift = kshift;
  il.segcnt = at<int32_t>(ws, R.segcnt);
  il.counts = at<int32_t>(ws, R.counts);
  il.offsets = at<int32_t>(ws, R.offsets);
  il.tile_base = at<int32_t>(ws, R.tile_base);
  il.perm = at<int32_t>(ws, R.perm);
  il.rank = at<int32_t>(ws, R.rank);
  il.farlen_tok = at<int32_t>(ws, R.far_tok);
  il.farlen_slot = at<int32_t>(ws, R.far_slot);
  il.items = at<focus_item_t>(ws, R.items);
  il.cost = at<int32_t>(ws, R.cost);
  il.order = at<int32_t>(ws, R.order);
  il.n_items = at<int32_t>(ws, R.n_items);
  il.max_items = R.max_items;
  il.err = err;
  return il;
}

void index_out(const IndexLaunch& il, focus_index_t* out) {
  out->counts = il.counts;
  out->offsets = il.offsets;
  out->perm = il.perm;
  out->rank = il.rank;
  out->farlen_tok = il.farlen_tok;
  out->farlen_slot = il.farlen_slot;
  out->items = il.items;
  out->order = il.order;
  out->n_items = il.n_items;
  out->max_items = il.max_items;
  out->w_eff = il.w_eff;
}

bool index_ok(const focus_index_t& x) {
  return x.perm && x.farlen_tok && x.farlen_slot && x.items && x.order && x.n_items;
}

// Group-pass arguments for one index (entries or pairs).
void group_args(AttnArgs& a, const focus_index_t& x, int m, int kshift, void* O_part, float* lse_part) {
  a.perm = x.perm;
  a.farlen_slot = x.farlen_slot;
  a.items = x.items;
  a.order = x.order;
  a.n_items = x.n_items;
  a.m = m;
  a.kshift = kshift;
  a.O_far = O_part;
  a.lse_far = lse_part;
}

// Streams and events focus_layer_fwd_host uses to overlap its copies with
// compute, created once per device (the library allocates no memory for them).
constexpr int kMaxChunks = 8;
struct HostPipe {
  cudaStream_t copy_in = nullptr, copy_out = nullptr;
  cudaEvent_t start = nullptr, inputs = nullptr, done = nullptr;
  cudaEvent_t chunk_in[kMaxChunks] = {}, chunk_out[kMaxChunks] = {};
  bool ready = false;
};
HostPipe g_pipe[64];

focus_status_t pipe_setup(HostPipe** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FOCUS_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  HostPipe& hp = g_pipe[dev];
  if (!hp.ready) {
    auto ev = [](cudaEvent_t* e) { return cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess; };
    bool ok = cudaStreamCreateWithFlags(&hp.copy_in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&hp.copy_out, cudaStreamNonBlocking) == cudaSuccess &&
              ev(&hp.start) && ev(&hp.inputs) && ev(&hp.done);
    for (int c = 0; ok && c < kMaxChunks; ++c) ok = ev(&hp.chunk_in[c]) && ev(&hp.chunk_out[c]);
    if (!ok) return FOCUS_ERR_CUDA;
    hp.ready = true;
  }
  *out = &hp;
  return FOCUS_OK;
}

}  // namespace
}  // namespace focus

using namespace focus;

extern "C" {

int32_t focus_abi_version(void) { return FOCUS_ABI_VERSION; }

const char* focus_status_string(focus_status_t s) {
  switch (s) {
    case FOCUS_OK: return "ok";
    case FOCUS_ERR_INVALID_ARG: return "invalid argument";
    case FOCUS_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case FOCUS_ERR_WORKSPACE: return "workspace too small";
    case FOCUS_ERR_CUDA: return "CUDA error";
    case FOCUS_ERR_TIMEOUT: return "device wait timed out";
    case FOCUS_ERR_BAD_GROUP_ID: return "group id outside [0, K)";
  }
  return "unknown status";
}

size_t focus_workspace_bytes(const focus_params_t* p) {
  if (!params_ok(p)) return 0;
  return layout_of(p).total;
}

focus_status_t focus_workspace_init(void* ws, void* stream) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1))) return FOCUS_ERR_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(ws, 0, kAlign, static_cast<cudaStream_t>(stream)));
}

static focus_status_t assign_impl(const focus_params_t* p, int k, const void* h, const void* W,
                                  const void* C, int32_t* gid, int* err, void* stream) {
  if (focus_status_t s = ensure_setup()) return s;
  AssignLaunch al{h, W, C, gid, p->B, p->n, p->D, p->d_g, p->K, p->A, k, err, nullptr, sm_count()};
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (p->dtype == FOCUS_F32) {
    if (!(p->d_g == 16 || p->d_g == 32 || p->d_g == 64 || p->d_g == 128)) return FOCUS_ERR_UNSUPPORTED;
    return cuda_status(launch_assign_f32(al, st));
  }
  if (!(p->d_g == 32 || p->d_g == 64 || p->d_g == 128)) return FOCUS_ERR_UNSUPPORTED;
  if (p->A * p->d_g > 512 || p->D % 8 != 0) return FOCUS_ERR_UNSUPPORTED;
  const int ncol = p->A * p->d_g;
  al.tile_rows = assign_tile_rows(p->B * p->n, ncol, al.num_sms);
  CUtensorMap tm_h, tm_w;
  if (!make_map(&tm_h, h, p->D, static_cast<uint64_t>(p->B) * p->n, 1, al.tile_rows, 2) ||
      !make_map(&tm_w, W, p->D, ncol, 1, ncol < 256 ? ncol : 256, 2))
    return FOCUS_ERR_CUDA;
  return cuda_status(launch_assign_bf16(al, &tm_h, &tm_w, st));
}

focus_status_t focus_assign(const focus_params_t* p, const void* h, const void* W, const void* C,
                            int32_t* gid, void* ws, size_t ws_bytes, void* stream) {
  if (!params_ok(p)) return FOCUS_ERR_INVALID_ARG;
  if (!h || !W || !C || !gid || !aligned16(h) || !aligned16(W) || !aligned16(C) || !aligned16(gid))
    return FOCUS_ERR_INVALID_ARG;
  if (focus_status_t s = check_ws(p, ws, ws_bytes)) return s;
  return assign_impl(p, 1, h, W, C, gid, at<int>(ws, layout_of(p).err), stream);
}

focus_status_t focus_build_index(const focus_params_t* p, const int32_t* gid,
                                 focus_index_t* idx_out, void* ws, size_t ws_bytes, void* stream) {
  if (!params_ok(p) || !gid || !idx_out || !aligned16(gid)) return FOCUS_ERR_INVALID_ARG;
  if (focus_status_t s = check_ws(p, ws, ws_bytes)) return s;
  if (focus_status_t s = ensure_setup()) return s;
  const Layout L = layout_of(p);
  IndexLaunch il{};
  il.gid = gid;
  il.P = p->B * p->A;
  il.A = p->A;
  il.n = p->n;
  il.K = p->K;
  il.w_eff = p->w > 1 ? p->w : 1;
  il.segcnt = at<int32_t>(ws, L.segcnt);
  il.counts = at<int32_t>(ws, L.counts);
  il.offsets = at<int32_t>(ws, L.offsets);
  il.tile_base = at<int32_t>(ws, L.tile_base);
  il.perm = at<int32_t>(ws, L.perm);
  il.rank = at<int32_t>(ws, L.rank);
  il.farlen_tok = at<int32_t>(ws, L.far_tok);
  il.farlen_slot = at<int32_t>(ws, L.far_slot);
  il.items = at<focus_item_t>(ws, L.items);
  il.cost = at<int32_t>(ws, L.cost);
  il.order = at<int32_t>(ws, L.order);
  il.n_items = at<int32_t>(ws, L.n_items);
  il.max_items = L.max_items;
  il.err = at<int>(ws, L.err);
  const focus_status_t s = cuda_status(launch_build_index(il, static_cast<cudaStream_t>(stream)));
  if (s != FOCUS_OK) return s;
  idx_out->counts = il.counts;
  idx_out->offsets = il.offsets;
  idx_out->perm = il.perm;
  idx_out->rank = il.rank;
  idx_out->farlen_tok = il.farlen_tok;
  idx_out->farlen_slot = il.farlen_slot;
  idx_out->items = il.items;
  idx_out->order = il.order;
  idx_out->n_items = il.n_items;
  idx_out->max_items = il.max_items;
  idx_out->w_eff = il.w_eff;
  return FOCUS_OK;
}

static focus_status_t attention_common(const focus_params_t* p, const void* Q, const void* K,
                                       const void* V, void* O, float* lse, void* ws,
                                       size_t ws_bytes) {
  if (!params_ok(p)) return FOCUS_ERR_INVALID_ARG;
  if (!Q || !K || !V || !O || !aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) ||
      (lse && !aligned16(lse)))
    return FOCUS_ERR_INVALID_ARG;
  if (!(p->d == 64 || p->d == 128)) return FOCUS_ERR_UNSUPPORTED;
  // tensor-map row coordinates are 32-bit
  if (static_cast<long long>(p->B) * p->H * p->n + kTileM >= (1LL << 31)) return FOCUS_ERR_UNSUPPORTED;
  if (focus_status_t s = check_ws(p, ws, ws_bytes)) return s;
  return ensure_setup();
}

focus_status_t focus_attention_fwd_timed(const focus_params_t* p, const void* Q, const void* K,
                                         const void* V, const focus_index_t* idx, void* O,
                                         float* lse_opt, void* ws, size_t ws_bytes, void* stream,
                                         void* const* events) {
  if (!idx || !idx->perm || !idx->farlen_tok || !idx->farlen_slot || !idx->items || !idx->order ||
      !idx->n_items)
    return FOCUS_ERR_INVALID_ARG;
  if (params_ok(p) && (idx->max_items != layout_of(p).max_items || idx->w_eff != (p->w > 1 ? p->w : 1)))
    return FOCUS_ERR_INVALID_ARG;
  if (focus_status_t s = attention_common(p, Q, K, V, O, lse_opt, ws, ws_bytes)) return s;
  const Layout L = layout_of(p);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  AttnArgs a = attn_args(p, Q, K, V, O, lse_opt, ws, L);
  a.perm = idx->perm;
  a.farlen_tok = idx->farlen_tok;
  a.farlen_slot = idx->farlen_slot;
  a.items = idx->items;
  a.order = idx->order;
  a.n_items = idx->n_items;
  auto mark = [&](int i) {
    return events ? cudaEventRecord(static_cast<cudaEvent_t>(events[i]), st) : cudaSuccess;
  };
  if (p->dtype == FOCUS_F32) {
    cudaError_t e = mark(0);
    if (e == cudaSuccess) e = mark(1);
    if (e == cudaSuccess) e = launch_attn_simt_f32(a, p->d, kModeGroup, L.max_items, st);
    if (e == cudaSuccess) e = mark(2);
    if (e == cudaSuccess) e = launch_attn_simt_f32(a, p->d, kModeLocal, 0, st);
    if (e == cudaSuccess) e = mark(3);
    return cuda_status(e);
  }
  void* Ks = at<void>(ws, L.Ks);
  void* Vs = at<void>(ws, L.Vs);
  cudaError_t e = mark(0);
  if (e == cudaSuccess) e = launch_permute_kv_bf16(K, V, Ks, Vs, idx->perm, p->B, p->H_kv, p->n, p->n, 0, p->d, p->A, st);
  if (e == cudaSuccess) e = mark(1);
  if (e != cudaSuccess) return FOCUS_ERR_CUDA;
  CUtensorMap tq, tk, tv, tks, tvs, to, tof;
  const uint64_t planes = static_cast<uint64_t>(p->B) * p->H_kv;
  const uint64_t qplanes = static_cast<uint64_t>(p->B) * p->H;
  if (!make_map(&tq, Q, p->d, p->n, qplanes, 128, 3) ||
      !make_map(&tk, K, p->d, p->n, planes, 128, 3) || !make_map(&tv, V, p->d, p->n, planes, 128, 3) ||
      !make_map(&tks, Ks, p->d, p->n, planes, 128, 3) || !make_map(&tvs, Vs, p->d, p->n, planes, 128, 3) ||
      !make_map(&to, O, p->d, p->n, qplanes, 128, 3) ||
      !make_map(&tof, a.O_far, p->d, p->n, qplanes, 128, 3))
    return FOCUS_ERR_CUDA;
  const int sms = sm_count();
  // group pass: Q rows are gathered through perm from a 2-D view with one-row boxes
  // group pass: Q rows are gathered through perm, and O_far rows scattered
  // back to token positions, through 2-D views with one-row boxes
  CUtensorMap tqg, tofs;
  if (!make_map(&tqg, Q, p->d, qplanes * p->n, 1, 1, 2) ||
      !make_map(&tofs, a.O_far, p->d, qplanes * p->n + kTileM, 1, 1, 2))
    return FOCUS_ERR_CUDA;
  e = launch_attn_tc_bf16(a, &tqg, &tks, &tvs, &tofs, &tof, p->d, kModeGroup, L.max_items, sms, st);
  if (e == cudaSuccess) e = mark(2);
  if (e == cudaSuccess) e = launch_attn_tc_bf16(a, &tq, &tk, &tv, &to, &tof, p->d, kModeLocal, 0, sms, st);
  if (e == cudaSuccess) e = mark(3);
  return cuda_status(e);
}

focus_status_t focus_attention_fwd(const focus_params_t* p, const void* Q, const void* K,
                                   const void* V, const focus_index_t* idx, void* O, float* lse_opt,
                                   void* ws, size_t ws_bytes, void* stream) {
  return focus_attention_fwd_timed(p, Q, K, V, idx, O, lse_opt, ws, ws_bytes, stream, nullptr);
}


focus_status_t focus_dense_causal_fwd(const focus_params_t* p, const void* Q, const void* K,
                                      const void* V, void* O, float* lse_opt, void* ws,
                                      size_t ws_bytes, void* stream) {
  if (focus_status_t s = attention_common(p, Q, K, V, O, lse_opt, ws, ws_bytes)) return s;
  const Layout L = layout_of(p);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  AttnArgs a = attn_args(p, Q, K, V, O, lse_opt, ws, L);
  a.w = p->n;
  if (p->dtype == FOCUS_F32) return cuda_status(launch_attn_simt_f32(a, p->d, kModeDense, 0, st));
  CUtensorMap tq, tk, tv, to;
  const uint64_t planes = static_cast<uint64_t>(p->B) * p->H_kv;
  const uint64_t qplanes = static_cast<uint64_t>(p->B) * p->H;
  if (!make_map(&tq, Q, p->d, p->n, qplanes, 128, 3) ||
      !make_map(&tk, K, p->d, p->n, planes, 128, 3) || !make_map(&tv, V, p->d, p->n, planes, 128, 3) ||
      !make_map(&to, O, p->d, p->n, qplanes, 128, 3))
    return FOCUS_ERR_CUDA;
  return cuda_status(launch_attn_tc_bf16(a, &tq, &tk, &tv, &to, &to, p->d, kModeDense, 0, sm_count(), st));
}

focus_status_t focus_test_attention_wait_limit(const focus_params_t* p, const void* Q, const void* K,
                                               const void* V, void* O, void* ws, size_t ws_bytes,
                                               uint64_t wait_ns, void* stream) {
  if (!params_ok(p) || wait_ns == 0 || wait_ns > kWaitLimitNs) return FOCUS_ERR_INVALID_ARG;
  if (p->dtype != FOCUS_BF16) return FOCUS_ERR_UNSUPPORTED;
  if (focus_status_t s = attention_common(p, Q, K, V, O, nullptr, ws, ws_bytes)) return s;
  const Layout L = layout_of(p);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  AttnArgs a = attn_args(p, Q, K, V, O, nullptr, ws, L);
  a.w = p->n;
  a.wait_ns = wait_ns;
  a.hold_first_q = 1;
  CUtensorMap tq, tk, tv, to;
  const uint64_t planes = static_cast<uint64_t>(p->B) * p->H_kv;
  const uint64_t qplanes = static_cast<uint64_t>(p->B) * p->H;
  if (!make_map(&tq, Q, p->d, p->n, qplanes, 128, 3) ||
      !make_map(&tk, K, p->d, p->n, planes, 128, 3) || !make_map(&tv, V, p->d, p->n, planes, 128, 3) ||
      !make_map(&to, O, p->d, p->n, qplanes, 128, 3))
    return FOCUS_ERR_CUDA;
  return cuda_status(launch_attn_tc_bf16(a, &tq, &tk, &tv, &to, &to, p->d, kModeDense, 0, sm_count(), st));
}

focus_status_t focus_attention_two_call_fwd(const focus_params_t* p, const void* Q, const void* K,
                                            const void* V, const focus_index_t* idx, void* O,
                                            float* lse_opt, void* ws, size_t ws_bytes, void* stream) {
  if (!idx || !idx->perm || !idx->farlen_tok || !idx->farlen_slot || !idx->items || !idx->order ||
      !idx->n_items)
    return FOCUS_ERR_INVALID_ARG;
  if (params_ok(p) && (idx->max_items != layout_of(p).max_items || idx->w_eff != (p->w > 1 ? p->w : 1)))
    return FOCUS_ERR_INVALID_ARG;
  if (focus_status_t s = attention_common(p, Q, K, V, O, lse_opt, ws, ws_bytes)) return s;
  const Layout L = layout_of(p);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  AttnArgs a = attn_args(p, Q, K, V, O, lse_opt, ws, L);
  a.perm = idx->perm;
  a.farlen_tok = idx->farlen_tok;
  a.farlen_slot = idx->farlen_slot;
  a.items = idx->items;
  a.order = idx->order;
  a.n_items = idx->n_items;
  // call 2 of the pair: a plain sliding-window attention (the dense mode with
  // the Focus window) writing O and its own LSE
  AttnArgs win = a;
  win.lse = at<float>(ws, L.lse_loc);
  CombineLaunch cl{O, win.lse, a.O_far, a.lse_far, idx->farlen_tok, lse_opt,
                   p->B, p->H, p->H_kv, p->A, p->n, p->d};
  cudaError_t e;
  if (p->dtype == FOCUS_F32) {
    e = launch_attn_simt_f32(a, p->d, kModeGroup, L.max_items, st);
    if (e == cudaSuccess) e = launch_attn_simt_f32(win, p->d, kModeDense, 0, st);
    if (e == cudaSuccess) e = launch_lse_combine(cl, p->dtype, st);
    return cuda_status(e);
  }
  void* Ks = at<void>(ws, L.Ks);
  void* Vs = at<void>(ws, L.Vs);
  e = launch_permute_kv_bf16(K, V, Ks, Vs, idx->perm, p->B, p->H_kv, p->n, p->n, 0, p->d, p->A, st);
  if (e != cudaSuccess) return FOCUS_ERR_CUDA;
  CUtensorMap tq, tk, tv, tks, tvs, to, tqg, tofs;
  const uint64_t planes = static_cast<uint64_t>(p->B) * p->H_kv;
  const uint64_t qplanes = static_cast<uint64_t>(p->B) * p->H;
  if (!make_map(&tq, Q, p->d, p->n, qplanes, 128, 3) ||
      !make_map(&tk, K, p->d, p->n, planes, 128, 3) || !make_map(&tv, V, p->d, p->n, planes, 128, 3) ||
      !make_map(&tks, Ks, p->d, p->n, planes, 128, 3) || !make_map(&tvs, Vs, p->d, p->n, planes, 128, 3) ||
      !make_map(&to, O, p->d, p->n, qplanes, 128, 3) ||
      !make_map(&tqg, Q, p->d, qplanes * p->n, 1, 1, 2) ||
      !make_map(&tofs, a.O_far, p->d, qplanes * p->n + kTileM, 1, 1, 2))
    return FOCUS_ERR_CUDA;
  const int sms = sm_count();
  e = launch_attn_tc_bf16(a, &tqg, &tks, &tvs, &tofs, &tofs, p->d, kModeGroup, L.max_items, sms, st);
  if (e == cudaSuccess) e = launch_attn_tc_bf16(win, &tq, &tk, &tv, &to, &to, p->d, kModeDense, 0, sms, st);
  if (e == cudaSuccess) e = launch_lse_combine(cl, p->dtype, st);
  return cuda_status(e);
}

focus_status_t focus_layer_fwd_host(const focus_params_t* p, const void* host_h,
                                    const void* host_W, const void* host_C, const void* host_Q,
                                    const void* host_K, const void* host_V, void* host_O,
                                    void* d_h, void* d_W, void* d_C, void* d_Q, void* d_K,
                                    void* d_V, void* d_O, int32_t* d_gid, void* ws,
                                    size_t ws_bytes, void* stream) {
  if (!params_ok(p)) return FOCUS_ERR_INVALID_ARG;
  if (!host_h || !host_W || !host_C || !host_Q || !host_K || !host_V || !host_O)
    return FOCUS_ERR_INVALID_ARG;
  if (!d_h || !d_W || !d_C || !d_Q || !d_K || !d_V || !d_O || !d_gid) return FOCUS_ERR_INVALID_ARG;
  if (focus_status_t s = ensure_setup()) return s;
  HostPipe* pp = nullptr;
  if (focus_status_t s = pipe_setup(&pp)) return s;
  const size_t es = elt_size(p->dtype);
  const size_t nb = static_cast<size_t>(p->B) * p->n;
  const size_t bytes_h = nb * p->D * es;
  const size_t bytes_W = static_cast<size_t>(p->A) * p->d_g * p->D * es;
  const size_t bytes_C = static_cast<size_t>(p->A) * p->K * p->d_g * es;
  const size_t bytes_Q = nb * p->H * p->d * es;
  const size_t bytes_KV = nb * p->H_kv * p->d * es;
  // Q/K/V (and O) move in KV-head chunks so each chunk's attention starts as
  // soon as its inputs land and its O goes back while later chunks compute.
  // Head slices are contiguous when B = 1, and with A = 1 every chunk shares
  // the one index; otherwise the layer runs as one chunk.
  int chunks = 1;
  if (p->B == 1 && p->A == 1)
    for (int c = kMaxChunks; c > 1; --c)
      if (p->H_kv % c == 0) { chunks = c; break; }
  focus_params_t pc = *p;
  pc.H = p->H / chunks;
  pc.H_kv = p->H_kv / chunks;
  const size_t cq = bytes_Q / chunks, ckv = bytes_KV / chunks;
  auto ptr = [](const void* b, size_t off) { return static_cast<const char*>(b) + off; };
  auto mptr = [](void* b, size_t off) { return static_cast<char*>(b) + off; };
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // host -> device, all on the copy-in stream, ordered after the caller's work
  if (cudaEventRecord(pp->start, st) != cudaSuccess || cudaStreamWaitEvent(pp->copy_in, pp->start, 0) != cudaSuccess)
    return FOCUS_ERR_CUDA;
  const struct { void* dst; const void* src; size_t n; } up[] = {
      {d_h, host_h, bytes_h}, {d_W, host_W, bytes_W}, {d_C, host_C, bytes_C}};
  for (const auto& c : up)
    if (cudaMemcpyAsync(c.dst, c.src, c.n, cudaMemcpyHostToDevice, pp->copy_in) != cudaSuccess)
      return FOCUS_ERR_CUDA;
  if (cudaEventRecord(pp->inputs, pp->copy_in) != cudaSuccess) return FOCUS_ERR_CUDA;
  for (int c = 0; c < chunks; ++c) {
    if (cudaMemcpyAsync(mptr(d_Q, c * cq), ptr(host_Q, c * cq), cq, cudaMemcpyHostToDevice, pp->copy_in) != cudaSuccess ||
        cudaMemcpyAsync(mptr(d_K, c * ckv), ptr(host_K, c * ckv), ckv, cudaMemcpyHostToDevice, pp->copy_in) != cudaSuccess ||
        cudaMemcpyAsync(mptr(d_V, c * ckv), ptr(host_V, c * ckv), ckv, cudaMemcpyHostToDevice, pp->copy_in) != cudaSuccess ||
        cudaEventRecord(pp->chunk_in[c], pp->copy_in) != cudaSuccess)
      return FOCUS_ERR_CUDA;
  }
  // assign and index once h, W, C are in
  if (cudaStreamWaitEvent(st, pp->inputs, 0) != cudaSuccess) return FOCUS_ERR_CUDA;
  focus_status_t s = focus_assign(p, d_h, d_W, d_C, d_gid, ws, ws_bytes, stream);
  if (s) return s;
  focus_index_t idx{};
  s = focus_build_index(p, d_gid, &idx, ws, ws_bytes, stream);
  if (s) return s;
  // attention per chunk on the caller's stream, O back on the copy-out stream
  for (int c = 0; c < chunks; ++c) {
    if (cudaStreamWaitEvent(st, pp->chunk_in[c], 0) != cudaSuccess) return FOCUS_ERR_CUDA;
    s = focus_attention_fwd(&pc, mptr(d_Q, c * cq), mptr(d_K, c * ckv), mptr(d_V, c * ckv), &idx,
                            mptr(d_O, c * cq), nullptr, ws, ws_bytes, stream);
    if (s) return s;
    if (cudaEventRecord(pp->chunk_out[c], st) != cudaSuccess ||
        cudaStreamWaitEvent(pp->copy_out, pp->chunk_out[c], 0) != cudaSuccess ||
        cudaMemcpyAsync(mptr(host_O, c * cq), mptr(d_O, c * cq), cq, cudaMemcpyDeviceToHost, pp->copy_out) != cudaSuccess)
      return FOCUS_ERR_CUDA;
  }
  // the caller's stream completes after the last copy back
  if (cudaEventRecord(pp->done, pp->copy_out) != cudaSuccess || cudaStreamWaitEvent(st, pp->done, 0) != cudaSuccess)
    return FOCUS_ERR_CUDA;
  return FOCUS_OK;
}

// ------------------------------------------------------ top-k membership ---

size_t focus_workspace_bytes_topk(const focus_params_t* p, int32_t k) {
  if (!topk_ok(p, k)) return 0;
  return layout_topk(p, k).total;
}

focus_status_t focus_assign_topk(const focus_params_t* p, int32_t k, const void* h, const void* W,
                                 const void* C, int32_t* gid, void* ws, size_t ws_bytes,
                                 void* stream) {
  if (!topk_ok(p, k)) return params_ok(p) && (k == 1 || k == 2) ? FOCUS_ERR_UNSUPPORTED : FOCUS_ERR_INVALID_ARG;
  if (!h || !W || !C || !gid || !aligned16(h) || !aligned16(W) || !aligned16(C) || !aligned16(gid))
    return FOCUS_ERR_INVALID_ARG;
  if (focus_status_t s = check_ws_topk(p, k, ws, ws_bytes)) return s;
  return assign_impl(p, k, h, W, C, gid, at<int>(ws, layout_topk(p, k).err), stream);
}

focus_status_t focus_build_index_topk(const focus_params_t* p, int32_t k, const int32_t* gid,
                                      focus_index_topk_t* idx_out, void* ws, size_t ws_bytes,
                                      void* stream) {
  if (!topk_ok(p, k)) return params_ok(p) && (k == 1 || k == 2) ? FOCUS_ERR_UNSUPPORTED : FOCUS_ERR_INVALID_ARG;
  if (!gid || !idx_out || !aligned16(gid)) return FOCUS_ERR_INVALID_ARG;
  if (focus_status_t s = check_ws_topk(p, k, ws, ws_bytes)) return s;
  if (focus_status_t s = ensure_setup()) return s;
  const LayoutTopk L = layout_topk(p, k);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int P = p->B * p->A, w_eff = p->w > 1 ? p->w : 1;
  int* err = at<int>(ws, L.err);
  focus_index_topk_t out{};
  out.k = k;
  if (L.split) {
    int32_t* vg = at<int32_t>(ws, L.vgid);
    int32_t* fsub = at<int32_t>(ws, L.far_sub);
    int32_t* fa = at<int32_t>(ws, L.far_any);
    if (launch_split_ids(gid, P, p->n, p->K, vg, err, st) != cudaSuccess) return FOCUS_ERR_CUDA;
    const IndexLaunch ie = index_launch(ws, L.ent, vg, P, p->A, L.m, p->K * p->K, w_eff, 1, err);
    if (launch_build_index_split(ie, p->K, fsub, st) != cudaSuccess) return FOCUS_ERR_CUDA;
    if (launch_far_any(ie.farlen_tok, P, p->n, fa, st) != cudaSuccess) return FOCUS_ERR_CUDA;
    index_out(ie, &out.entry);
    out.split = 1;
    out.farlen_sub = fsub;
    out.far_tok = fa;
    *idx_out = out;
    return FOCUS_OK;
  }
  const IndexLaunch ie = index_launch(ws, L.ent, gid, P, p->A, L.m, p->K, w_eff, k == 2 ? 1 : 0, err);
  if (launch_build_index(ie, st) != cudaSuccess) return FOCUS_ERR_CUDA;
  index_out(ie, &out.entry);
  if (k == 2) {
    int32_t* pg = at<int32_t>(ws, L.pair_gid);
    int32_t* fa = at<int32_t>(ws, L.far_any);
    if (launch_pair_ids(gid, P, p->n, p->K, pg, err, st) != cudaSuccess) return FOCUS_ERR_CUDA;
    const IndexLaunch ip = index_launch(ws, L.pair, pg, P, p->A, p->n, L.Kp, w_eff, 0, err);
    if (launch_build_index(ip, st) != cudaSuccess) return FOCUS_ERR_CUDA;
    if (launch_far_any(ie.farlen_tok, P, p->n, fa, st) != cudaSuccess) return FOCUS_ERR_CUDA;
    index_out(ip, &out.pair);
    out.pair_gid = pg;
    out.far_tok = fa;
  } else {
    out.far_tok = ie.farlen_tok;    // one entry per token: its farlen is the flag
  }
  *idx_out = out;
  return FOCUS_OK;
}

focus_status_t focus_attention_topk_fwd_timed(const focus_params_t* p, const void* Q, const void* K,
                                              const void* V, const focus_index_topk_t* idx,
                                              void* O, float* lse_opt, void* ws, size_t ws_bytes,
                                              void* stream, void* const* events) {
  if (!idx || !(idx->k == 1 || idx->k == 2)) return FOCUS_ERR_INVALID_ARG;
  const int k = idx->k;
  if (!topk_ok(p, k)) return params_ok(p) ? FOCUS_ERR_UNSUPPORTED : FOCUS_ERR_INVALID_ARG;
  const LayoutTopk L = layout_topk(p, k);
  const int w_eff = p->w > 1 ? p->w : 1;
  if (!index_ok(idx->entry) || !idx->far_tok || idx->entry.max_items != L.ent.max_items ||
      idx->entry.w_eff != w_eff)
    return FOCUS_ERR_INVALID_ARG;
  if ((idx->split != 0) != L.split || (L.split && !idx->farlen_sub)) return FOCUS_ERR_INVALID_ARG;
  if (k == 2 && !L.split &&
      (!index_ok(idx->pair) || idx->pair.max_items != L.pair.max_items || idx->pair.w_eff != w_eff))
    return FOCUS_ERR_INVALID_ARG;
  if (!Q || !K || !V || !O || !aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) ||
      (lse_opt && !aligned16(lse_opt)))
    return FOCUS_ERR_INVALID_ARG;
  if (!(p->d == 64 || p->d == 128)) return FOCUS_ERR_UNSUPPORTED;
  const uint64_t qplanes = static_cast<uint64_t>(p->B) * p->H;
  const uint64_t planes = static_cast<uint64_t>(p->B) * p->H_kv;
  // tensor-map rows and the row scatter's targets are 32-bit
  if (static_cast<long long>(qplanes) * L.m + kTileM >= (1LL << 31)) return FOCUS_ERR_UNSUPPORTED;
  if (focus_status_t s = check_ws_topk(p, k, ws, ws_bytes)) return s;
  if (focus_status_t s = ensure_setup()) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  auto mark = [&](int i) {
    return events ? cudaEventRecord(static_cast<cudaEvent_t>(events[i]), st) : cudaSuccess;
  };
  Layout none{};
  none.err = L.err;
  none.O_far = L.O_far;
  none.lse_far = L.lse_far;
  const AttnArgs base = attn_args(p, Q, K, V, O, lse_opt, ws, none);
  void* O_far = at<void>(ws, L.O_far);
  float* lse_far = at<float>(ws, L.lse_far);
  void* O_e = k == 2 ? at<void>(ws, L.O_e) : O_far;
  float* lse_e = k == 2 ? at<float>(ws, L.lse_e) : lse_far;
  void* O_p = at<void>(ws, L.O_p);
  float* lse_p = at<float>(ws, L.lse_p);
  AttnArgs ge = base;
  group_args(ge, idx->entry, L.m, k == 2 ? 1 : 0, O_e, lse_e);
  if (L.split) {
    ge.farlen_sub = idx->farlen_sub;
    ge.nsub = p->K - 1;
    ge.offsets = idx->entry.offsets;
  }
  // the pair pass subtracts the pairs the entry pass visits twice; the split
  // index visits none twice
  const bool pair_pass = k == 2 && !L.split;
  AttnArgs gp = base;
  if (pair_pass) group_args(gp, idx->pair, p->n, 0, O_p, lse_p);
  AttnArgs lo = base;
  lo.farlen_tok = idx->far_tok;
  MergeLaunch ml{O_e, lse_e, pair_pass ? O_p : nullptr, pair_pass ? lse_p : nullptr, idx->entry.farlen_tok,
                 pair_pass ? idx->pair.farlen_tok : nullptr, O_far, lse_far,
                 p->B, p->H, p->H_kv, p->A, p->n, p->d};
  cudaError_t e = mark(0);
  if (p->dtype == FOCUS_F32) {
    if (e == cudaSuccess) e = mark(1);
    if (e == cudaSuccess) e = launch_attn_simt_f32(ge, p->d, kModeGroup, L.ent.max_items, st);
    if (e == cudaSuccess) e = mark(2);
    if (pair_pass && e == cudaSuccess) e = launch_attn_simt_f32(gp, p->d, kModeGroup, L.pair.max_items, st);
    if (k == 2 && e == cudaSuccess) e = launch_topk_merge(ml, p->dtype, st);
    if (e == cudaSuccess) e = mark(3);
    if (e == cudaSuccess) e = launch_attn_simt_f32(lo, p->d, kModeLocal, 0, st);
    if (e == cudaSuccess) e = mark(4);
    return cuda_status(e);
  }
  void* Ks = at<void>(ws, L.Ks);
  void* Vs = at<void>(ws, L.Vs);
  const int sms = sm_count();
  if (e == cudaSuccess)
    e = launch_permute_kv_bf16(K, V, Ks, Vs, idx->entry.perm, p->B, p->H_kv, p->n, L.m, ge.kshift, p->d, p->A, st);
  if (e == cudaSuccess) e = mark(1);
  if (e != cudaSuccess) return FOCUS_ERR_CUDA;
  // entry pass: Q rows gathered by token, partial rows scattered by entry
  CUtensorMap tqg, tks, tvs, tofs;
  if (!make_map(&tqg, Q, p->d, qplanes * p->n, 1, 1, 2) ||
      !make_map(&tks, Ks, p->d, L.m, planes, 128, 3) || !make_map(&tvs, Vs, p->d, L.m, planes, 128, 3) ||
      !make_map(&tofs, O_e, p->d, qplanes * L.m + kTileM, 1, 1, 2))
    return FOCUS_ERR_CUDA;
  e = launch_attn_tc_bf16(ge, &tqg, &tks, &tvs, &tofs, &tofs, p->d, L.split ? kModeGroupSplit : kModeGroup,
                          L.ent.max_items, sms, st);
  if (e == cudaSuccess) e = mark(2);
  if (e == cudaSuccess && k == 2 && !pair_pass) e = launch_topk_merge(ml, p->dtype, st);
  if (e == cudaSuccess && pair_pass) {
    // pair pass over the same K/V buffers, re-sorted by pair (the entry pass
    // is done with them: same stream)
    CUtensorMap pks, pvs, pofs;
    e = launch_permute_kv_bf16(K, V, Ks, Vs, idx->pair.perm, p->B, p->H_kv, p->n, p->n, 0, p->d, p->A, st);
    if (e != cudaSuccess) return FOCUS_ERR_CUDA;
    if (!make_map(&pks, Ks, p->d, p->n, planes, 128, 3) || !make_map(&pvs, Vs, p->d, p->n, planes, 128, 3) ||
        !make_map(&pofs, O_p, p->d, qplanes * p->n + kTileM, 1, 1, 2))
      return FOCUS_ERR_CUDA;
    e = launch_attn_tc_bf16(gp, &tqg, &pks, &pvs, &pofs, &pofs, p->d, kModeGroup, L.pair.max_items, sms, st);
    if (e == cudaSuccess) e = launch_topk_merge(ml, p->dtype, st);
  }
  if (e == cudaSuccess) e = mark(3);
  if (e != cudaSuccess) return FOCUS_ERR_CUDA;
  CUtensorMap tq, tk, tv, to, tof;
  if (!make_map(&tq, Q, p->d, p->n, qplanes, 128, 3) ||
      !make_map(&tk, K, p->d, p->n, planes, 128, 3) || !make_map(&tv, V, p->d, p->n, planes, 128, 3) ||
      !make_map(&to, O, p->d, p->n, qplanes, 128, 3) || !make_map(&tof, O_far, p->d, p->n, qplanes, 128, 3))
    return FOCUS_ERR_CUDA;
  e = launch_attn_tc_bf16(lo, &tq, &tk, &tv, &to, &tof, p->d, kModeLocal, 0, sms, st);
  if (e == cudaSuccess) e = mark(4);
  return cuda_status(e);
}

focus_status_t focus_attention_topk_fwd(const focus_params_t* p, const void* Q, const void* K,
                                        const void* V, const focus_index_topk_t* idx, void* O,
                                        float* lse_opt, void* ws, size_t ws_bytes, void* stream) {
  return focus_attention_topk_fwd_timed(p, Q, K, V, idx, O, lse_opt, ws, ws_bytes, stream, nullptr);
}

// ------------------------------------------------ Sinkhorn soft assignment ---

static size_t sinkhorn_layout(const focus_params_t* p, size_t* u, size_t* v, size_t* part,
                              size_t* ticket) {
  const size_t P = static_cast<size_t>(p->B) * p->A;
  const int rpc = sinkhorn_rows_per_chunk(p->n);
  const size_t chunks = (static_cast<size_t>(p->n) + rpc - 1) / rpc;
  size_t o = align_up(kAlign);                       // error word
  *u = o;
  o = align_up(o + P * p->n * 4);
  *v = o;
  o = align_up(o + P * p->K * 4);
  *part = o;
  o = align_up(o + P * chunks * p->K * 8);
  *ticket = o;
  o = align_up(o + P * 4);
  return o;
}

size_t focus_sinkhorn_workspace_bytes(const focus_params_t* p) {
  if (!params_ok(p)) return 0;
  size_t u, v, part, ticket;
  return sinkhorn_layout(p, &u, &v, &part, &ticket);
}

focus_status_t focus_assign_scores(const focus_params_t* p, const void* h, const void* W,
                                   const void* C, float* S, void* ws, size_t ws_bytes,
                                   void* stream) {
  if (!params_ok(p)) return FOCUS_ERR_INVALID_ARG;
  if (!h || !W || !C || !S || !aligned16(h) || !aligned16(W) || !aligned16(C) || !aligned16(S))
    return FOCUS_ERR_INVALID_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1))) return FOCUS_ERR_INVALID_ARG;
  if (ws_bytes < focus_sinkhorn_workspace_bytes(p)) return FOCUS_ERR_WORKSPACE;
  if (focus_status_t s = ensure_setup()) return s;
  AssignLaunch al{h, W, C, nullptr, p->B, p->n, p->D, p->d_g, p->K, p->A, 1, at<int>(ws, 0), S, sm_count()};
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (p->dtype == FOCUS_F32) {
    if (!(p->d_g == 16 || p->d_g == 32 || p->d_g == 64 || p->d_g == 128)) return FOCUS_ERR_UNSUPPORTED;
    return cuda_status(launch_assign_f32(al, st));
  }
  if (!(p->d_g == 32 || p->d_g == 64 || p->d_g == 128)) return FOCUS_ERR_UNSUPPORTED;
  if (p->A * p->d_g > 512 || p->D % 8 != 0) return FOCUS_ERR_UNSUPPORTED;
  const int ncol = p->A * p->d_g;
  al.tile_rows = assign_tile_rows(p->B * p->n, ncol, al.num_sms);
  CUtensorMap tm_h, tm_w;
  if (!make_map(&tm_h, h, p->D, static_cast<uint64_t>(p->B) * p->n, 1, al.tile_rows, 2) ||
      !make_map(&tm_w, W, p->D, ncol, 1, ncol < 256 ? ncol : 256, 2))
    return FOCUS_ERR_CUDA;
  return cuda_status(launch_assign_bf16(al, &tm_h, &tm_w, st));
}

focus_status_t focus_sinkhorn_fwd(const focus_params_t* p, int32_t iters, float tau, const float* S,
                                  float* G, void* ws, size_t ws_bytes, void* stream) {
  if (!params_ok(p)) return FOCUS_ERR_INVALID_ARG;
  if (iters < 1 || iters > 10000 || !(std::isfinite(tau) && tau > 0.f)) return FOCUS_ERR_INVALID_ARG;
  if (!S || !G || !aligned16(S) || !aligned16(G)) return FOCUS_ERR_INVALID_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1))) return FOCUS_ERR_INVALID_ARG;
  size_t u, v, part, ticket;
  if (ws_bytes < sinkhorn_layout(p, &u, &v, &part, &ticket)) return FOCUS_ERR_WORKSPACE;
  if (focus_status_t s = ensure_setup()) return s;
  SinkhornLaunch L{S, G, at<float>(ws, u), at<float>(ws, v), at<float2>(ws, part), at<int>(ws, ticket),
                   p->B * p->A, p->n, p->K, 1.f / tau, at<int>(ws, 0), sm_count()};
  return cuda_status(launch_sinkhorn(L, iters, static_cast<cudaStream_t>(stream)));
}

// ------------------------------------------------------------- backward ---

struct BwdLayout {
  size_t delta, dq, dk, dv, qs, dos, ks, vs, lse_s, delta_s, kv_order, total;
};

static BwdLayout backward_layout(const focus_params_t* p) {
  BwdLayout L{};
  const size_t qrows = static_cast<size_t>(p->B) * p->H * p->n;
  const size_t krows = static_cast<size_t>(p->B) * p->H_kv * p->n;
  size_t o = align_up(kAlign);                       // error word
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes);
    return at;
  };
  L.delta = take(qrows * 4);
  L.dq = take(qrows * p->d * 4);
  L.dk = take(krows * p->d * 4);
  L.dv = take(krows * p->d * 4);
  if (p->dtype == FOCUS_BF16) {
    // the group kernels' operands in index order
    L.qs = take(qrows * p->d * 2);
    L.dos = take(qrows * p->d * 2);
    L.ks = take(krows * p->d * 2);
    L.vs = take(krows * p->d * 2);
    L.lse_s = take(qrows * 4);
    L.delta_s = take(qrows * 4);
    // the far dK/dV kernel's units (128 key slots of one KV head), longest first
    L.kv_order = take(static_cast<size_t>(p->B) * p->H_kv * ((p->n + 127) / 128) * 4);
  }
  L.total = o;
  return L;
}

size_t focus_backward_workspace_bytes(const focus_params_t* p) {
  if (!params_ok(p)) return 0;
  return backward_layout(p).total;
}

focus_status_t focus_attention_bwd(const focus_params_t* p, const void* Q, const void* K,
                                   const void* V, const void* O, const void* dO, const float* lse,
                                   const focus_index_t* idx, void* dQ, void* dK, void* dV, void* ws,
                                   size_t ws_bytes, void* stream) {
  if (!params_ok(p)) return FOCUS_ERR_INVALID_ARG;
  if (!idx || !idx->perm || !idx->farlen_tok || !idx->farlen_slot || !idx->offsets || !idx->items ||
      !idx->order || !idx->n_items)
    return FOCUS_ERR_INVALID_ARG;
  if (idx->max_items != layout_of(p).max_items || idx->w_eff != (p->w > 1 ? p->w : 1))
    return FOCUS_ERR_INVALID_ARG;
  const void* ptrs[] = {Q, K, V, O, dO, lse, dQ, dK, dV};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return FOCUS_ERR_INVALID_ARG;
  if (!(p->d == 64 || p->d == 128)) return FOCUS_ERR_UNSUPPORTED;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1))) return FOCUS_ERR_INVALID_ARG;
  const BwdLayout BL = backward_layout(p);
  if (ws_bytes < BL.total) return FOCUS_ERR_WORKSPACE;
  if (focus_status_t s = ensure_setup()) return s;
  BwdArgs a{};
  a.Q = Q;
  a.K = K;
  a.V = V;
  a.O = O;
  a.dO = dO;
  a.lse = lse;
  a.delta = at<float>(ws, BL.delta);
  a.dq_far = at<float>(ws, BL.dq);
  a.dk_far = at<float>(ws, BL.dk);
  a.dv_far = at<float>(ws, BL.dv);
  a.err = at<int>(ws, 0);
  a.dQ = dQ;
  a.dK = dK;
  a.dV = dV;
  a.perm = idx->perm;
  a.farlen_tok = idx->farlen_tok;
  a.farlen_slot = idx->farlen_slot;
  a.offsets = idx->offsets;
  a.items = idx->items;
  a.order = idx->order;
  a.n_items = idx->n_items;
  a.B = p->B;
  a.H = p->H;
  a.H_kv = p->H_kv;
  a.n = p->n;
  a.d = p->d;
  a.A = p->A;
  a.groups = p->K;
  a.w = idx->w_eff;
  a.scale = p->scale;
  a.scale_log2 = p->scale * 1.4426950408889634f;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (p->dtype == FOCUS_F32) return cuda_status(launch_attn_bwd(a, p->dtype, idx->max_items, st));
  // bf16: tensor cores
  const uint64_t qplanes = static_cast<uint64_t>(p->B) * p->H;
  const uint64_t planes = static_cast<uint64_t>(p->B) * p->H_kv;
  if (static_cast<long long>(qplanes) * p->n >= (1LL << 31)) return FOCUS_ERR_UNSUPPORTED;
  void* Qs = at<void>(ws, BL.qs);
  void* dOs = at<void>(ws, BL.dos);
  void* Ks = at<void>(ws, BL.ks);
  void* Vs = at<void>(ws, BL.vs);
  a.lse_sorted = at<float>(ws, BL.lse_s);
  a.delta_sorted = at<float>(ws, BL.delta_s);
  a.ticket = at<int>(ws, 0) + 1;   // the word after the error word
  a.kv_order = at<int32_t>(ws, BL.kv_order);
  // tile maps over the sorted copies (group kernels) and the inputs (window kernels)
  CUtensorMap qs3, dos3, ks3, vs3, q3, do3, k3, v3;
  if (!make_map(&qs3, Qs, p->d, p->n, qplanes, 128, 3) || !make_map(&dos3, dOs, p->d, p->n, qplanes, 128, 3) ||
      !make_map(&ks3, Ks, p->d, p->n, planes, 128, 3) || !make_map(&vs3, Vs, p->d, p->n, planes, 128, 3) ||
      !make_map(&q3, Q, p->d, p->n, qplanes, 128, 3) || !make_map(&do3, dO, p->d, p->n, qplanes, 128, 3) ||
      !make_map(&k3, K, p->d, p->n, planes, 128, 3) || !make_map(&v3, V, p->d, p->n, planes, 128, 3))
    return FOCUS_ERR_CUDA;
  // Delta comes with the index-order copy of Q, dO, LSE (one read of dO)
  cudaError_t e = launch_bwd_permute_q(a, Qs, dOs, at<float>(ws, BL.lse_s), at<float>(ws, BL.delta_s), st);
  if (e == cudaSuccess)
    e = launch_permute_kv_bf16(K, V, Ks, Vs, idx->perm, p->B, p->H_kv, p->n, p->n, 0, p->d, p->A, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(a.ticket, 0, sizeof(int), st);
  if (e == cudaSuccess) e = launch_attn_bwd_tc(a, &qs3, &dos3, &ks3, &vs3, &q3, &do3, &k3, &v3, idx->max_items, sm_count(), st);
  return cuda_status(e);
}

focus_status_t focus_check_errors(void* ws, void* stream) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1))) return FOCUS_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return FOCUS_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FOCUS_ERR_CUDA;
  if (word == 0) return FOCUS_OK;
  if (cudaMemset(ws, 0, sizeof(int)) != cudaSuccess) return FOCUS_ERR_CUDA;
  if (word & kErrTimeout) return FOCUS_ERR_TIMEOUT;
  if (word & kErrBadGroup) return FOCUS_ERR_BAD_GROUP_ID;
  return FOCUS_ERR_CUDA;
}

}  // extern "C"
