/*
 * focus.h -- C ABI of the Focus attention hot path on one NVIDIA GB300 (sm_103a).
 *
 * Focus keeps, for causal attention, only the token pairs that matter:
 * pairs inside a local window, and far pairs whose two tokens fall in the
 * same learned group; every other pair is skipped, and softmax stays exact
 * over the kept pairs.  Sources (page titles and sections):
 *   "Focus: Learning Which Attention Pairs Matter", section 2.1 (centroids,
 *     projection, local + group-gated far attention), section 2.2 (hard
 *     top-k assignment at inference; far pairs of different groups skipped;
 *     pair count O(n^2/K + n*w)), section 3.3 (local-window + in-group causal
 *     decomposition).
 *   "Why Attend to Everything? Focus is the Key", section 2.1 (exact softmax
 *     preserved), section 2.3 (hard assignment, two FlashAttention calls).
 *
 * The hot path is three calls, issued in order on one stream:
 *   focus_assign        hidden states -> group id per token (top-1 centroid)
 *   focus_build_index   group ids -> (group, position) sorted index + work list
 *   focus_attention_fwd Q, K, V, index -> O over the kept pairs only
 * Around it: focus_dense_causal_fwd (the dense comparator),
 * focus_attention_two_call_fwd (the pages' two-call strategy, a comparator),
 * focus_layer_fwd_host (the layer from host buffers), the top-k membership
 * calls (*_topk, k = 2), the Sinkhorn soft assignment (focus_assign_scores,
 * focus_sinkhorn_fwd), the backward (focus_attention_bwd) and
 * focus_build_index_static (the index without a workspace).
 *
 * Conventions shared by every call
 *   - All tensor pointers are DEVICE pointers to row-major contiguous arrays,
 *     16-byte aligned, owned by the caller.  The library allocates nothing,
 *     keeps no state beyond a per-process cache of kernel attributes, and
 *     never synchronises except in focus_check_errors.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   - `ws` is caller-owned device scratch of at least focus_workspace_bytes(p)
 *     bytes, 256-byte aligned.  It holds the device error word, the index and
 *     attention temporaries; one workspace serves one stream at a time.
 *   - Argument errors are reported synchronously as a status with nothing
 *     launched.  Launch failures give FOCUS_ERR_CUDA.  Errors found on the
 *     device (a group id outside [0, K), a bounded wait that ran out) set bits
 *     of the device error word and are reported by focus_check_errors.  No
 *     call traps, asserts, aborts or throws across this boundary.
 *
 * Shapes (notation of the pages plus standard attention names)
 *   B batch, H query heads, H_kv key/value heads (H % H_kv == 0),
 *   n tokens, d head dim, D hidden size, d_g projection dim, K centroids,
 *   A independent assignments (1: one group id per token shared by all heads;
 *   H_kv: one per key/value head), w local window (pair kept when i - j < w;
 *   w = 0 keeps the same pairs as w = 1 because a token always shares its own
 *   group), scale softmax scale (1/sqrt(d) in the usual setting).
 *   Query head h reads key/value head kv = h * H_kv / H (integer division) and
 *   assignment a = (A == 1 ? 0 : kv).
 */
#ifndef FOCUS_H_
#define FOCUS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FOCUS_ABI_VERSION 3   /* 2: adds the top-k membership calls; 3: the split top-2 index layout */

#if defined(__GNUC__)
#define FOCUS_API __attribute__((visibility("default")))
#else
#define FOCUS_API
#endif

/* Query rows per group-pass work item; the work list is built for this height. */
#define FOCUS_TILE_M 128
/* Keys per attention tile; the longest-first schedule counts cost in these. */
#define FOCUS_TILE_N 128
/* Largest supported number of centroids K. */
#define FOCUS_MAX_K 4096
/* Largest supported sequence length n. */
#define FOCUS_MAX_N (1 << 20)

typedef enum {
  FOCUS_OK = 0,
  FOCUS_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad shape or value   */
  FOCUS_ERR_UNSUPPORTED = 2,   /* valid request with no kernel (dtype, d, ...)  */
  FOCUS_ERR_WORKSPACE = 3,     /* ws_bytes < focus_workspace_bytes(p)           */
  FOCUS_ERR_CUDA = 4,          /* a CUDA runtime/launch call failed             */
  FOCUS_ERR_TIMEOUT = 5,       /* device: a bounded wait ran out                */
  FOCUS_ERR_BAD_GROUP_ID = 6   /* device: a group id outside [0, K)             */
} focus_status_t;

typedef enum { FOCUS_F32 = 0, FOCUS_BF16 = 1 } focus_dtype_t;

/* Problem description; every call takes the same struct. */
typedef struct {
  int32_t B, H, H_kv, n, d, D, d_g, K, A, w;
  float scale;
  int32_t dtype; /* focus_dtype_t: element type of h, W, C, Q, K, V and O */
} focus_params_t;

/* One group-pass work item: query rows = sorted slots row0 .. row0+rows-1 of
 * assignment (b, a), all in group g; keys = the first `keys` slots of that
 * group, starting at slot key0 (= offsets[g]). */
typedef struct {
  int32_t b, a, g, row0, rows, keys, key0, pad;
} focus_item_t;

/* Device pointers into the workspace, filled by focus_build_index.
 * Arrays are indexed [(b * A + a) * len + i]. */
typedef struct {
  int32_t* counts;       /* [B*A][K]   tokens per group                         */
  int32_t* offsets;      /* [B*A][K+1] exclusive scan of counts                 */
  int32_t* perm;         /* [B*A][n]   sorted slot -> token position            */
  int32_t* rank;         /* [B*A][n]   token position -> sorted slot            */
  int32_t* farlen_tok;   /* [B*A][n]   per position: same-group tokens j<=i-w   */
  int32_t* farlen_slot;  /* [B*A][n]   the same, per sorted slot                */
  focus_item_t* items;   /* [max_items] work list, canonical (b, a, g, row0)    */
  int32_t* order;        /* [max_items] longest-first schedule over items       */
  int32_t* n_items;      /* [1]        number of valid entries in items/order   */
  int32_t max_items;     /* host-side capacity of items/order                   */
  int32_t w_eff;         /* window the index was built for (max(w, 1))          */
} focus_index_t;

/* Bytes of device workspace the calls below need for problem p (0 if p is
 * invalid).  Pure host arithmetic. */
FOCUS_API size_t focus_workspace_bytes(const focus_params_t* p);

/* Clears the device error word at the start of ws (an async memset on
 * `stream`).  Call once after allocating a workspace, before the first call
 * that uses it; focus_check_errors clears the word again after each report. */
FOCUS_API focus_status_t focus_workspace_init(void* ws, void* stream);

/* Group assignment ("Focus: Learning Which Attention Pairs Matter" 2.1, 2.2;
 * "Why Attend to Everything?" 2.3).  For each token i of batch b and each
 * assignment a: p = W[a] h[b,i] (no bias, accumulated and kept in fp32),
 * s_k = p . C[a,k] in fp32, gid[b,a,i] = argmax_k s_k, lowest k on ties.
 *   h   [B, n, D]      dtype          W [A, d_g, D] dtype     C [A, K, d_g] dtype
 *   gid [B, A, n]      int32 output
 * bf16 runs the projection on the tensor cores (fp32 accumulate) and needs
 * D % 8 == 0, d_g in {32, 64, 128} and A*d_g <= 512; with d_g = 64 and K <= 64
 * the scores run there too, from p split exactly into three bf16 parts
 * (exact products, fp32 accumulation in the tensor core's order), otherwise
 * as fp32 FMAs.  f32 runs everything in fp32 on the CUDA cores and needs d_g
 * in {16, 32, 64, 128}.  Other shapes give FOCUS_ERR_UNSUPPORTED. */
FOCUS_API focus_status_t focus_assign(const focus_params_t* p, const void* h, const void* W,
                            const void* C, int32_t* gid, void* ws, size_t ws_bytes,
                            void* stream);

/* Group-sorted index ("Focus: Learning Which Attention Pairs Matter" 2.2: far
 * pairs of different groups are skipped, so each group's tokens are gathered).
 * Stable counting sort of tokens by (group, position) per (b, a), farlen per
 * token, and the group-pass work list in canonical order plus a longest-first
 * order.  gid [B, A, n] int32 device input.  *idx_out (host struct) receives
 * device pointers into ws; they stay valid while ws is not reused by another
 * focus_build_index.  A gid outside [0, K) is clamped for safety and flagged
 * as FOCUS_ERR_BAD_GROUP_ID in the device error word. */
FOCUS_API focus_status_t focus_build_index(const focus_params_t* p, const int32_t* gid,
                                 focus_index_t* idx_out, void* ws, size_t ws_bytes,
                                 void* stream);

/* Bytes of the fixed device scratch behind focus_build_index_static. */
#define FOCUS_INDEX_STATIC_SCRATCH_BYTES (1u << 20)

/* focus_build_index with no workspace and no allocation.  The papers have no
 * counterpart: this is a deployment entry point for callers that cannot
 * allocate device memory when they build the index (a process whose device
 * footprint is fixed at start-up, or one that wants the index without the
 * attention workspace).  Same operation and bit-identical outputs as
 * focus_build_index.
 *   gid  [B, A, n] int32 device input, 16-byte aligned.
 *   idx  host struct, in/out.  On entry counts, offsets, perm, rank,
 *        farlen_tok, farlen_slot, items, order and n_items are caller-owned
 *        device buffers (16-byte aligned) sized as documented for
 *        focus_index_t, and max_items is the capacity of items and order,
 *        at least B*A*(ceil(n / FOCUS_TILE_M) + min(K, n)).  On return
 *        max_items holds that bound and w_eff the window, so the index can be
 *        passed to focus_attention_fwd like one from focus_build_index.
 *   err  device int32 error word, 256-byte aligned (focus_check_errors(err,
 *        stream) reads and clears it).  It must hold 0 before the first call;
 *        kernels only OR bits into it (FOCUS_ERR_BAD_GROUP_ID as in
 *        focus_build_index).
 * The sort's scratch (per-segment histograms, tile bases, item costs:
 * 4*(B*A*ceil(n/1024)*K + B*A*(K+1) + max_items) bytes plus alignment) comes
 * from one fixed device array of FOCUS_INDEX_STATIC_SCRATCH_BYTES per device;
 * a larger problem returns FOCUS_ERR_WORKSPACE before anything is launched.
 * Nothing in that array has to start at zero.  All calls on a device share it,
 * so calls whose kernels may overlap (other streams, other host threads) race:
 * order them, e.g. on one stream.  The first call on each device looks up the
 * array's address and sets kernel attributes; make that call before capturing
 * a stream.  Returns FOCUS_ERR_INVALID_ARG for a bad p, pointer or capacity. */
FOCUS_API focus_status_t focus_build_index_static(const focus_params_t* p, const int32_t* gid,
                                                  focus_index_t* idx, int32_t* err,
                                                  void* stream);

/* Focus attention over the kept pairs ("Focus: Learning Which Attention Pairs
 * Matter" 2.1, 2.2, 3.3; "Why Attend to Everything?" 2.1, 2.3).  Row i of head h
 * attends to key j iff j <= i and (i - j < w or g_i == g_j), with
 * softmax(scale * q_i . k_j) exact over that set.
 *   Q [B, H, n, d], K/V [B, H_kv, n, d] dtype, O [B, H, n, d] dtype output,
 *   lse_opt [B, H, n] fp32 natural-log sum-exp of the scaled scores, or NULL.
 * idx must come from focus_build_index with the same p and ws.  d in {64, 128}.
 * The call runs a group pass (far same-group keys, rows in sorted order) and a
 * local pass (window keys, natural order) that merges both partial softmaxes. */
FOCUS_API focus_status_t focus_attention_fwd(const focus_params_t* p, const void* Q, const void* K,
                                   const void* V, const focus_index_t* idx, void* O,
                                   float* lse_opt, void* ws, size_t ws_bytes, void* stream);

/* focus_attention_fwd that also records four caller-created CUDA events
 * (cudaEvent_t, passed as void*) on `stream`: events[0] before the K/V sort
 * copy, events[1] before the group pass, events[2] before the local pass and
 * events[3] after it, so a caller can time each kernel.  events == NULL is
 * exactly focus_attention_fwd.  Same arguments and errors otherwise. */
FOCUS_API focus_status_t focus_attention_fwd_timed(const focus_params_t* p, const void* Q,
                                                   const void* K, const void* V,
                                                   const focus_index_t* idx, void* O,
                                                   float* lse_opt, void* ws, size_t ws_bytes,
                                                   void* stream, void* const* events);

/* Ordinary causal attention (every j <= i kept) with the same kernels and
 * layouts as the local pass: the dense comparator for the speedup figure.
 * Ignores p->w, p->K, p->A.  Same tensors and rules as focus_attention_fwd. */
FOCUS_API focus_status_t focus_dense_causal_fwd(const focus_params_t* p, const void* Q, const void* K,
                                      const void* V, void* O, float* lse_opt, void* ws,
                                      size_t ws_bytes, void* stream);

/* Test hook for the device-side failure path; not part of the method.  Runs
 * the bf16 dense causal kernel of focus_dense_causal_fwd with every bounded
 * wait limited to wait_ns nanoseconds (1 <= wait_ns <= 10^9) and with its Q
 * load warp withholding the first Q tile, so the first S product's wait runs
 * out: the kernel raises its abort flag, lets the copies it issued land, frees
 * TMEM and exits.  focus_check_errors(ws) then reports FOCUS_ERR_TIMEOUT (and
 * clears it); O holds no result.  Arguments, layouts and the workspace as
 * focus_dense_causal_fwd; bf16 only (FOCUS_ERR_UNSUPPORTED otherwise). */
FOCUS_API focus_status_t focus_test_attention_wait_limit(const focus_params_t* p, const void* Q,
                                                 const void* K, const void* V, void* O, void* ws,
                                                 size_t ws_bytes, uint64_t wait_ns, void* stream);

/* The two-call comparator: the same operation and tensors as
 * focus_attention_fwd, run the way the pages run it ("Why Attend to
 * Everything? Focus is the Key" 2.3; "Focus: Learning Which Attention Pairs
 * Matter" 3.3): an in-group causal call (the group pass, writing its partial
 * to ws), a standalone sliding-window attention call writing O and its LSE,
 * and a separate log-sum-exp combine that updates O in place.
 * focus_attention_fwd instead merges inside the local pass; this call exists
 * to measure that fusion.  idx, ws, errors and lse_opt as focus_attention_fwd
 * (lse_opt must not alias ws). */
FOCUS_API focus_status_t focus_attention_two_call_fwd(const focus_params_t* p, const void* Q,
                                                      const void* K, const void* V,
                                                      const focus_index_t* idx, void* O,
                                                      float* lse_opt, void* ws, size_t ws_bytes,
                                                      void* stream);

/* The whole layer from HOST buffers: copies h, W, C, Q, K, V from host memory
 * (pinned, for the copies to overlap) into the caller's device buffers, runs
 * assign -> index -> attention on `stream`, and copies O back to host memory.
 * When B = 1 and A = 1, Q/K/V and O move in KV-head chunks on two
 * library-owned streams (created once per device): each chunk's attention
 * starts when its inputs have landed and its O returns while later chunks
 * compute.  Everything is ordered after the caller's earlier work on `stream`
 * and completes on `stream`.  d_* are device buffers of the sizes above;
 * d_gid is [B, A, n] int32.  Returns after enqueueing; synchronise the stream
 * (or call focus_check_errors) before reading host_O.  Calls on one device
 * share the internal streams: do not overlap two calls. */
FOCUS_API focus_status_t focus_layer_fwd_host(const focus_params_t* p,
                                    const void* host_h, const void* host_W, const void* host_C,
                                    const void* host_Q, const void* host_K, const void* host_V,
                                    void* host_O,
                                    void* d_h, void* d_W, void* d_C, void* d_Q, void* d_K,
                                    void* d_V, void* d_O, int32_t* d_gid,
                                    void* ws, size_t ws_bytes, void* stream);

/* ----------------------------------------------------- top-k membership ---
 * "Focus: Learning Which Attention Pairs Matter" 2.2 (each token is
 * hard-assigned to its top-k groups at inference) and 3.3; "Why Attend to
 * Everything? Focus is the Key" 2.3 (K = 4, k = 2 in its experiment).  With k
 * groups per token, row i attends to key j iff j <= i and (i - j < w or the
 * group sets of i and j intersect); softmax is exact over that set and a key
 * that shares several groups with the query still counts once.  k is 1 or 2;
 * k = 1 is the top-1 operation above.  Memberships are "entries": entry
 * e = i * k + c is token i's c-th best group.
 *
 * Index layout for k memberships, all device pointers into ws, arrays
 * indexed [(b * A + a) * len + x]:
 *   entry      focus_index_t over the n*k entries: counts/offsets per group,
 *              perm (sorted slot -> entry e), rank (entry -> slot),
 *              farlen_tok (per ENTRY: members of that entry's group at token
 *              positions j <= i - w), farlen_slot (the same per slot), and the
 *              group-pass work list; every length n there reads n*k.
 *   pair       k = 2 only: focus_index_t over tokens sorted by their group
 *              pair {a, b} (K (K - 1) / 2 pair ids, numbered (0,1), (0,2), ...,
 *              (0,K-1), (1,2), ...).  Its far members are the far keys that
 *              share BOTH groups with the query, which the entry pass counts
 *              twice; the attention call subtracts them once.
 *   pair_gid   k = 2: [B*A][n] pair id per token.
 *   far_tok    [B*A][n] 1 if token i has any far key, else 0.
 * k = 2 needs K (K - 1) / 2 <= FOCUS_MAX_K (K <= 91), else
 * FOCUS_ERR_UNSUPPORTED.
 *
 * Split layout (k = 2, K <= 8 and bf16 tensors; split = 1): no pair index.  The entry index
 * sorts the entries by virtual group v = g * K + o (g the entry's group, o the
 * token's other group), then by position, so counts/offsets have K * K (+1)
 * entries and each group g splits into K - 1 sub-runs (g, o').  farlen_sub
 * [B*A][2n][K-1] (by slot, column j = o' - (o' > g)) holds the slot's far
 * members in sub-run (g, o'), 0 for o' = o when o < g: a pair of tokens that
 * share both groups is visited once, in the smaller group's pass.  farlen_tok
 * and farlen_slot hold each entry's / slot's total over its sub-runs, and the
 * work list has one item per (row tile, sub-run): item.g = v, item.pad = j,
 * key0 = the sub-run's first slot. */
typedef struct {
  focus_index_t entry;
  focus_index_t pair;
  int32_t* pair_gid;
  int32_t* far_tok;
  int32_t k;
  int32_t split;         /* 1: split layout (see above), 0: entry + pair */
  int32_t* farlen_sub;   /* split layout only, else NULL */
} focus_index_topk_t;

/* Bytes of device workspace the top-k calls need for problem p and k (0 if p
 * or k is invalid or unsupported).  Pure host arithmetic.  The layout differs
 * from focus_workspace_bytes'; a top-k workspace serves only top-k calls. */
FOCUS_API size_t focus_workspace_bytes_topk(const focus_params_t* p, int32_t k);

/* Top-k assignment: as focus_assign, with the k best centroids per token.
 *   gid [B, A, n, k] int32 output: gid[b,a,i,0] the best centroid, [.., 1] the
 *   runner-up; among equal fp32 scores the lower index ranks first.
 * Shapes, dtypes and errors as focus_assign; ws is a top-k workspace. */
FOCUS_API focus_status_t focus_assign_topk(const focus_params_t* p, int32_t k, const void* h,
                                           const void* W, const void* C, int32_t* gid, void* ws,
                                           size_t ws_bytes, void* stream);

/* Top-k index: the entry index (stable counting sort of the n*k entries by
 * (group, entry), i.e. by (group, position)), farlen per entry and slot and
 * the work list; for k = 2 also the pair ids, the pair index and far_tok, or
 * for K <= 8 with bf16 tensors the split layout above.
 * gid [B, A, n, k] int32 device input; a token's k ids must differ.  A gid
 * outside [0, K), or two equal ids of one token, is clamped or refiled for
 * safety and flagged as FOCUS_ERR_BAD_GROUP_ID in the device error word.
 * *idx_out (host struct) receives device pointers into ws, valid until ws is
 * reused by another index build. */
FOCUS_API focus_status_t focus_build_index_topk(const focus_params_t* p, int32_t k,
                                                const int32_t* gid, focus_index_topk_t* idx_out,
                                                void* ws, size_t ws_bytes, void* stream);

/* Top-k Focus attention over the kept pairs.  Tensors, d, lse_opt and errors
 * as focus_attention_fwd; idx from focus_build_index_topk with the same p and
 * ws.  Runs: the group pass over entries (one partial per entry), for k = 2 a
 * group pass over pair ids and a merge that combines each token's two entry
 * partials minus its pair partial by log-sum-exp (split layout: no pair pass,
 * the merge adds the two entry partials), then the local pass that merges the
 * far partial with the window keys. */
FOCUS_API focus_status_t focus_attention_topk_fwd(const focus_params_t* p, const void* Q,
                                                  const void* K, const void* V,
                                                  const focus_index_topk_t* idx, void* O,
                                                  float* lse_opt, void* ws, size_t ws_bytes,
                                                  void* stream);

/* focus_attention_topk_fwd recording five caller-created CUDA events on
 * `stream` (NULL = none): events[0] before the entry K/V sort copy, [1] before
 * the entry group pass, [2] after it, [3] before the local pass (after the
 * pair pass and the merge), [4] after the local pass. */
FOCUS_API focus_status_t focus_attention_topk_fwd_timed(const focus_params_t* p, const void* Q,
                                                        const void* K, const void* V,
                                                        const focus_index_topk_t* idx, void* O,
                                                        float* lse_opt, void* ws, size_t ws_bytes,
                                                        void* stream, void* const* events);

/* --------------------------------------------- Sinkhorn soft assignment ---
 * The training-time assignment ("Focus: Learning Which Attention Pairs
 * Matter" 2.1, 2.3; "Why Attend to Everything? Focus is the Key" 2.2): tokens
 * are assigned softly to the K groups and Sinkhorn normalisation makes the
 * n x K assignment matrix doubly stochastic, so every group gets an equal
 * share of the tokens.  The pages give neither the temperature nor the number
 * of rounds: both are arguments.  For each (b, a), with X = S / tau,
 *   G = diag(e^u) exp(X) diag(e^v): every row of G sums to 1 and every column
 *   to n / K in the limit; T rounds of Sinkhorn-Knopp scaling, each round
 *   first the columns (to n / K) then the rows (to 1), from u = 0.
 * Both calls take a Sinkhorn workspace of focus_sinkhorn_workspace_bytes(p)
 * (256-byte aligned; error word first, as for the other calls). */
FOCUS_API size_t focus_sinkhorn_workspace_bytes(const focus_params_t* p);

/* All token-to-centroid scores: S[b,a,i,k] = (W[a] h[b,i]) . C[a,k], fp32
 * accumulate, as focus_assign computes them before its argmax.
 *   h, W, C as focus_assign; S [B, A, n, K] fp32 device output.
 * Shapes and errors as focus_assign. */
FOCUS_API focus_status_t focus_assign_scores(const focus_params_t* p, const void* h,
                                             const void* W, const void* C, float* S, void* ws,
                                             size_t ws_bytes, void* stream);

/* Sinkhorn forward: S [B, A, n, K] fp32 scores -> G [B, A, n, K] fp32 soft
 * assignment (G may be S: updated in place).  iters = T in [1, 10000],
 * tau > 0 finite, else FOCUS_ERR_INVALID_ARG.  Log-domain arithmetic in fp32.
 * For K <= 256 with K % 4 == 0 a round is one launch and one pass over S (the
 * row step fused with the next round's column step), plus one column pass up
 * front; other K take two passes and three launches per round. */
FOCUS_API focus_status_t focus_sinkhorn_fwd(const focus_params_t* p, int32_t iters, float tau,
                                            const float* S, float* G, void* ws, size_t ws_bytes,
                                            void* stream);

/* ------------------------------------------------------------- backward ---
 * Gradients of focus_attention_fwd over the kept pairs, for training or
 * fine-tuning a retrofitted model ("Why Attend to Everything? Focus is the
 * Key" 2.1: exact softmax over the kept pairs; "Focus: Learning Which
 * Attention Pairs Matter" 3.1).  With P_ij = exp(scale q_i.k_j - lse_i) on
 * kept pairs and Delta_i = dO_i . O_i:
 *   dV_j = sum_i P_ij dO_i,  dS_ij = P_ij (dO_i . v_j - Delta_i),
 *   dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i,
 * dK, dV summed over the query heads of each key/value head.
 *   Q, O, dO, dQ [B, H, n, d]; K, V, dK, dV [B, H_kv, n, d]: dtype of p,
 *   16-byte aligned; lse [B, H, n] fp32 from the forward call (lse_opt);
 *   idx from focus_build_index with the same p (in the forward workspace).
 * ws: a backward workspace of focus_backward_workspace_bytes(p) (error word
 * first; fp32 partials; for bf16 also index-ordered copies of Q, dO, K, V and
 * the far dK/dV kernel's work order).
 * bf16 runs on the tcgen05 tensor cores (bf16 products, fp32 accumulate and
 * softmax arithmetic); fp32 runs in fp32 on the CUDA cores.  d in {64, 128}.
 * Errors as focus_attention_fwd. */
FOCUS_API size_t focus_backward_workspace_bytes(const focus_params_t* p);

FOCUS_API focus_status_t focus_attention_bwd(const focus_params_t* p, const void* Q, const void* K,
                                             const void* V, const void* O, const void* dO,
                                             const float* lse, const focus_index_t* idx, void* dQ,
                                             void* dK, void* dV, void* ws, size_t ws_bytes,
                                             void* stream);

/* Synchronises `stream`, reads and clears the device error word in ws.
 * Returns FOCUS_OK, FOCUS_ERR_BAD_GROUP_ID, FOCUS_ERR_TIMEOUT or FOCUS_ERR_CUDA. */
FOCUS_API focus_status_t focus_check_errors(void* ws, void* stream);

/* Static description of a status code. */
FOCUS_API const char* focus_status_string(focus_status_t s);

/* FOCUS_ABI_VERSION of the loaded library. */
FOCUS_API int32_t focus_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FOCUS_H_ */
