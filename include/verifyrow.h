/*
 * verifyrow -- the data-parallel hot path of the speculative-decoding verify
 * step, for one NVIDIA GB300 (sm_103a).
 *
 * One verify window scores the next position and every draft token in one
 * pass ("Speculative decoding on RDNA", §01 figure "one speculative
 * window": k drafts, k + 1 verify rows), penalises every row against its own
 * history (§04), turns each row into the sampler's distribution (§03 "how
 * hipfire does it") and decides how many drafts to keep (§02 greedy, §03
 * rejection sampling; token trees from "One RDNA4 verify pass has slack for
 * about two dozen speculative tokens", "Spend the budget on a tree"; naive
 * sampling verify from "feat(dflash): developer-only online draft tuning",
 * notes under the spec-step listing).
 *
 * Conventions that hold for every entry point below.
 *   - Array arguments are DEVICE pointers owned by the caller, unless the
 *     argument is documented as a host pointer.  The library allocates no
 *     memory: its scratch is the caller's workspace `ws` of `ws_bytes`
 *     bytes (device memory, 256-byte aligned), sized by vr_workspace_bytes.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work
 *     is enqueued asynchronously; outputs are valid once the stream has
 *     reached that point.  No entry point synchronises unless it says so.
 *   - Kernels are launched with programmatic dependent launch.  Every input
 *     except the weights is read only after the kernel before it on the
 *     stream has completed.  The tensor-core projection requests its first
 *     weight blocks as soon as it starts, which is before that kernel ends
 *     when the kernel lets dependents launch early (griddepcontrol.
 *     launch_dependents); a kernel that does so must not write the weights.
 *   - Return value: VR_OK or a negative VR_ERR_* code.  Argument errors are
 *     detected on the host before anything is enqueued.  Errors that depend
 *     on device-resident data (a token outside the vocabulary, a parent
 *     array that is not topological) are recorded in a status word inside
 *     the workspace and make that window emit nothing (*out_n_emitted = 0);
 *     read them with vr_device_status.  Nothing traps on the device.
 *   - Rows and nodes.  A window verifies n_nodes draft nodes over
 *     rows = n_nodes + 1 rows.  Row 0 scores the current position; row 1+j
 *     scores the position after node j.  `parent` == NULL means a chain
 *     (node j hangs from node j-1); otherwise parent[j] is -1 (the root) or
 *     an earlier node.  Node j is checked against row(parent[j]).
 *   - Matrices are row-major.  weight: [vocab][hidden] bf16 bit patterns
 *     (the LM-head layout); act: [rows][hidden] float; logits:
 *     [rows][vocab] float.
 */
#ifndef VERIFYROW_H
#define VERIFYROW_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define VR_API __attribute__((visibility("default")))
#else
#define VR_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define VR_ABI_VERSION 1

/* status codes */
#define VR_OK 0
#define VR_ERR_ARG (-1)          /* a NULL, a size out of range, bad policy    */
#define VR_ERR_CUDA (-2)         /* a CUDA call or launch failed               */
#define VR_ERR_UNSUPPORTED (-3)  /* shape the kernels do not handle            */
#define VR_ERR_DEVICE (-4)       /* the device status word is set              */
#define VR_ERR_WORKSPACE (-5)    /* ws is NULL, misaligned or too small        */

/* device status word bits (vr_device_status) */
#define VR_DEV_BAD_TOKEN 1       /* a draft token outside [0, vocab)           */
#define VR_DEV_BAD_PARENT 2      /* parent[j] not in [-1, j)                   */
#define VR_DEV_BAD_QID 4         /* a draft candidate id outside [0, vocab)    */
#define VR_DEV_TIMEOUT 8         /* a bounded on-chip wait gave up             */

/* projection paths; chosen per weight matrix, never by row count */
#define VR_PATH_AUTO 0           /* = VR_PATH_TC                               */
#define VR_PATH_FFMA 1           /* CUDA-core multi-row GEMV (fp32 FMA)        */
#define VR_PATH_TC 2             /* tcgen05 tensor cores, exact 3-plane split  */
#define VR_PATH_TC_BATCH 3       /* tcgen05, rows as M in groups of 256, 2 planes */

/* limits */
#define VR_POOL 64               /* pool width ("Speculative decoding on RDNA" §03) */
#define VR_QCAND 8               /* draft candidates per draft row (same section)   */
#define VR_MAX_WINDOW_ROWS 64    /* rows of one request (k + 1 or nodes + 1)         */
#define VR_MAX_ROWS 1024         /* rows of one projection / batched call            */
#define VR_MAX_PENALTY_WINDOW 512
#define VR_MAX_REQUESTS 256

/*
 * Sampler and penalty settings of one request ("Speculative decoding on
 * RDNA" §03: temperature, top-k (20 when absent, all 64 pool entries when
 * 0), min-p, top-p; §04: repeat, presence and frequency penalties over the last
 * W tokens).  temperature == 0 means greedy.  Validation (VR_ERR_ARG):
 * temperature, min_p, top_p finite and temperature >= 0; repeat finite and
 * > 0; presence, frequency finite; 0 <= window <= VR_MAX_PENALTY_WINDOW.
 */
typedef struct vr_policy {
  float temperature;  /* 0 => greedy                                        */
  int32_t top_k;      /* < 0 absent => 20; 0 => 64 (whole pool); > 64 => 64 */
  float min_p;        /* <= 0 disables                                      */
  float top_p;        /* >= 1 disables                                      */
  float repeat;       /* 1 disables                                         */
  float presence;     /* 0 disables                                         */
  float frequency;    /* 0 disables                                         */
  int32_t window;     /* W; 0 disables every penalty                        */
} vr_policy;

/* One request of a batched call (host struct holding device pointers). */
typedef struct vr_request {
  int32_t n_nodes;          /* the request owns n_nodes + 1 consecutive rows  */
  const int32_t* tokens;    /* [n_nodes] draft tokens                         */
  const int32_t* parent;    /* [n_nodes] or NULL (chain)                      */
  const int32_t* q_ids;     /* [n_nodes][8] draft candidates or NULL          */
  const float* q_logits;    /* [n_nodes][8] their logits or NULL              */
  const int32_t* hist;      /* [hist_len] prompt || emitted so far            */
  int32_t hist_len;
  vr_policy policy;
  uint64_t seed;            /* request seed of the random stream              */
  uint64_t position;        /* |prompt || emitted| at the window start        */
  int32_t* out_ids;         /* [n_nodes + 1] emitted ids first; later entries unspecified */
  int32_t* out_accept;      /* [1] accepted drafts                            */
  int32_t* out_n_emitted;   /* [1] emitted ids (accepted + 1; 0 on error)     */
} vr_request;

/* ABI version (VR_ABI_VERSION) and a static text for a status code. */
VR_API int vr_abi_version(void);
VR_API const char* vr_status_string(int status);

/*
 * Workspace bytes for a call over `rows` rows (all requests together),
 * `hidden` and `vocab`.  One workspace may be reused by consecutive calls
 * on one stream; calls that may overlap need separate workspaces.
 * Errors: VR_ERR_ARG if out_bytes is NULL or a size is out of range.
 */
VR_API int vr_workspace_bytes(int rows, int hidden, int vocab, size_t* out_bytes);

/*
 * (a1) Multi-row verify projection ("Speculative decoding on RDNA" §01: the
 * weights are read once for all k + 1 rows; §02: multi-row projections sum
 * in the single-row order).
 *   logits[r][v] = sum_h weight[v][h] * act[r][h], fp32 accumulation.
 * Paths (chosen per weight matrix, never by row count):
 *   VR_PATH_TC (= AUTO): rows in groups of 32, activations split exactly into
 *     three bf16 planes (exact products); the weights stream once per group.
 *   VR_PATH_TC_BATCH: rows in groups of 256 as the MMA's M side, two bf16
 *     planes (16 significant bits, error below 2^-17 |a|); weights stream once
 *     per group.  For many rows (batched serving), where the tensor pipe sets
 *     the pace.
 *   VR_PATH_FFMA: CUDA-core FMAs, rows in passes of up to 8; a pass keeps
 *     its activations in shared memory (4 * hidden bytes per row), so hidden
 *     above 51200 returns VR_ERR_UNSUPPORTED on this path.
 * For a given path, hidden and vocab, the bits of row r do not depend on
 * `rows` or on the other rows' values, so a row computed inside an R-row
 * call is identical to the same row computed alone.
 * Accuracy against exact arithmetic: |error| <= 1e-3 * max(1, |logit|) on
 * every path for hidden up to 32768, and on VR_PATH_TC up to 65536 (the
 * tensor-core paths' fp32 accumulation error grows about linearly with
 * hidden; VR_PATH_TC_BATCH adds both planes in one accumulator and reaches
 * about 1.35 times that bound at 65536; VR_PATH_FFMA stays about a hundred
 * times below it).
 * rows in [1, VR_MAX_ROWS]; hidden a multiple of 8 in [8, 65536];
 * vocab in [1, 2^31 - 1].  path: VR_PATH_*.  Writes logits only.
 */
VR_API int vr_verify_project(const uint16_t* weight, const float* act, int rows, int hidden,
                      int vocab, int path, float* logits, void* ws, size_t ws_bytes,
                      void* stream);

/*
 * (a2) Per-row penalty prepass, in place ("Speculative decoding on RDNA"
 * §04): row r is penalised against H_r, the last W tokens of
 * (hist || tokens on the path root -> node r-1), i.e. for a chain
 * H_i = last W of (prompt || emitted || drafts[0..i)).  For each distinct
 * token t of H_r with count c (t outside [0, vocab) is ignored), in float32
 * operations rounded to nearest:
 *   x = logits[r][t]; if repeat != 1: x = x > 0 ? x / repeat : x * repeat;
 *   if frequency != 0: x -= (float)c * frequency; if presence != 0: x -= presence.
 * If q_logits is non-NULL the same is applied in place to the draft
 * candidates of node j (q_ids[j][0..8)) with H_row(parent[j]).  A policy with
 * window == 0 or all three penalties neutral leaves everything untouched.
 * rows = n_nodes + 1 <= VR_MAX_WINDOW_ROWS.
 */
VR_API int vr_verify_penalize(float* logits, int rows, int vocab, const int32_t* tokens,
                       const int32_t* parent, int n_nodes, const int32_t* hist, int hist_len,
                       const vr_policy* policy, const int32_t* q_ids, float* q_logits,
                       void* ws, size_t ws_bytes, void* stream);

/*
 * (a3) Candidate pool of every row: the first min(64, vocab) entries of the
 * row in the order (value descending, token id ascending), where every NaN
 * ranks below -inf and -0.0 below +0.0 ("Speculative decoding on RDNA" §03:
 * a 64-wide pool with a fixed tie order).  pool_ids/pool_vals:
 * [rows][64]; slots past min(64, vocab) get id -1 and value NaN.
 * pool_vals holds the logits' own bits.  pool_ids[r][0] is the row argmax.
 */
VR_API int vr_verify_select(const float* logits, int rows, int vocab, int32_t* pool_ids,
                     float* pool_vals, void* ws, size_t ws_bytes, void* stream);

/*
 * Batched top-K of float rows: the first k entries of each row in the pool
 * order above (value descending, token id ascending, NaN below -inf, -0.0
 * below +0.0).  The same select as vr_verify_select cut to k; it serves the
 * many-row top-K of a draft tuner ("feat(dflash): developer-only online
 * draft tuning", the re-grid top-K select measured at 15 rows x 248320,
 * K = 16, gated on byte identity with ties, NaN and -inf).
 * x [rows][vocab]; ids/vals [rows][k] (row stride k); k in [1, VR_POOL];
 * slots past min(k, vocab) get id -1 and value NaN; vals holds x's own bits.
 * rows in [1, VR_MAX_ROWS].  Scratch from ws as for vr_verify_select
 * (vr_workspace_bytes(rows, 8, vocab) suffices).
 */
VR_API int vr_topk(const float* x, int rows, int vocab, int k, int32_t* ids, float* vals,
                   void* ws, size_t ws_bytes, void* stream);

/*
 * vr_verify_select without a workspace.  The pages have no counterpart: this
 * entry point exists for callers that cannot give the library device memory
 * of its own (for example a plugin whose host application owns every device
 * allocation, or a process that must not grow its device footprint after
 * start-up).  Same inputs, outputs and results as vr_verify_select; the
 * select's intermediate candidates and its row counters live in a fixed
 * 1 MiB array compiled into the library, which every GPU that loads the
 * library keeps until exit.  Each call clears the counters with an
 * asynchronous memset on `stream` before its kernel.
 * Limits and rules:
 *   - rows <= VR_NOALLOC_SELECT_MAX_ROWS (else VR_ERR_UNSUPPORTED); any vocab;
 *   - the array is shared by all calls on a device and keeps the last call's
 *     contents; calls that overlap on the GPU race on it, so the caller must
 *     serialise them (one stream, one thread at a time);
 *   - the first call on each device looks the array's address up on that
 *     device (cudaGetSymbolAddress, the device must be current).  Under
 *     CUDA's lazy module loading (the default) that lookup is also what
 *     places the array, about 1 MiB, and the select's kernel code in that
 *     device's memory, so the device footprint grows once, at the first
 *     call.  Make that first call at start-up, before any stream capture on
 *     the device; later calls leave the device's free memory unchanged.
 * Calls no cudaMalloc, cudaFree or allocating library routine, on any call.
 */
#define VR_NOALLOC_SELECT_MAX_ROWS 32
VR_API int vr_verify_select_noalloc(const float* logits, int rows, int vocab, int32_t* pool_ids,
                                    float* pool_vals, void* stream);

/*
 * (a4) Sampler policy on given pools ("Speculative decoding on RDNA" §03):
 * pool_vals [rows][64] in pool order, pool_len valid entries per row.
 * All arithmetic is IEEE float32, each operation rounded to nearest, sums
 * sequential in pool order.  K = 20 if top_k absent, 64 if 0, else
 * min(top_k, 64), at most pool_len; greedy (temperature 0) keeps pool[0]
 * alone with weight 1; otherwise e_0 = 1, e_j = vexp((v_j - v_0) / T)
 * (0 for NaN or -inf, or an exponent below -87), then min-p cuts at the
 * first e_j < min_p, top-p keeps the shortest prefix whose running sum
 * reaches top_p * sum, and S is the sum of the kept weights.  vexp is a
 * Cody-Waite reduction plus a degree-7 Taylor polynomial in float32 +, -, x
 * only, so results are identical on every IEEE machine.
 * Outputs: out_m [rows] kept count, out_e [rows][64] (zeros past m),
 * out_S [rows].
 */
VR_API int vr_verify_policy(const float* pool_vals, int rows, int pool_len, const vr_policy* policy,
                     int32_t* out_m, float* out_e, float* out_S, void* stream);

/*
 * (a3)+(a4)+(a5) Pool, policy and acceptance on already-penalised logits.
 *   greedy: chain -> the longest prefix of drafts equal to the row argmax,
 *     then the argmax at the first mismatch or the bonus after the last row
 *     (§02); tree -> the deepest node whose whole path agrees with the
 *     argmax of each parent row (equal depths: the lower node index).
 *   sampled chain: rejection sampling (§03): accept d_i iff
 *     u1 * q_i(d_i) < p_i(d_i) (q_i(d_i) = 0: iff p_i(d_i) > 0); a rejected
 *     d_i is replaced by a sample of (p_i - q_i)+ renormalised (of p_i if
 *     that is all zero), which ends the window; after k acceptances draw the bonus from p_k.
 *     With q_ids/q_logits (penalised by the caller), q_i is the same policy
 *     on the 8 candidates of node i ordered like the pool.  Without them
 *     (q_ids == NULL: drafts proposed without probabilities, such as n-gram
 *     matches), q_i = delta(d_i) (§06 "N-gram takeovers"): d_i is accepted
 *     iff u1 < p_i(d_i), and the replacement is drawn from p_i with d_i
 *     removed.
 *   sampled tree: naive sampling descent: from the root draw y ~ p(row);
 *     move to the lowest-index child carrying y, else emit y and stop.
 * Draws: u = Philox4x64-10(counter = (position, row, purpose, 0),
 * key = (seed, 0)) word 0 >> 40, times 2^-24 (a float32); purpose 1 = accept
 * uniform, 2 = emitted draw; t = u * S picks the first j whose running sum
 * exceeds t.  The probabilities, accept test and residual are float32.
 * Outputs: out_ids [n_nodes + 1] (the emitted ids first; the entries after
 * them hold unspecified values), out_accept, out_n_emitted (= accepted + 1
 * >= 1; 0 if the device status was set).
 */
VR_API int vr_verify_sample_accept(const float* pen_logits, int rows, int vocab, const int32_t* tokens,
                            const int32_t* parent, int n_nodes, const int32_t* q_ids,
                            const float* q_logits, const vr_policy* policy, uint64_t seed,
                            uint64_t position, int32_t* out_ids, int32_t* out_accept,
                            int32_t* out_n_emitted, void* ws, size_t ws_bytes, void* stream);

/*
 * The whole window in one call: projection -> penalties -> pool -> policy ->
 * acceptance, enqueued on `stream` with no host synchronisation (kernels
 * only, so the call may be captured into a CUDA graph and replayed).
 * logits receives the raw projection.  If the policy has active penalties:
 * pen_logits (if non-NULL) receives the penalised rows and logits stays raw;
 * if pen_logits is NULL, logits is penalised in place.  q_logits is read
 * only (its penalised copy lives in ws).  Semantics as in the calls above.
 */
VR_API int vr_verify_window(const uint16_t* weight, const float* act, int rows, int hidden, int vocab,
                     int path, const int32_t* tokens, const int32_t* parent, int n_nodes,
                     const int32_t* q_ids, const float* q_logits, const int32_t* hist,
                     int hist_len, const vr_policy* policy, uint64_t seed, uint64_t position,
                     float* logits, float* pen_logits, int32_t* out_ids, int32_t* out_accept,
                     int32_t* out_n_emitted, void* ws, size_t ws_bytes, void* stream);

/*
 * Many independent requests in one call: their rows are stacked in `act`
 * (request b owns n_nodes_b + 1 consecutive rows, in the order of `reqs`)
 * and share one projection; penalties, pools, policies and acceptance run
 * per request with that request's policy, seed, position and history.
 * `reqs` is a HOST array of n_req descriptors; the call copies them into the
 * parameters of the kernels it enqueues (which store them into ws), so the
 * array may be reused or freed as soon as the call returns, and the call may
 * be captured into a CUDA graph (each replay uses the descriptors as they
 * were at capture).  total rows <= VR_MAX_ROWS, n_req <= VR_MAX_REQUESTS.
 * logits/pen_logits as in vr_verify_window.
 */
VR_API int vr_verify_window_batched(const uint16_t* weight, const float* act, int hidden, int vocab,
                             int path, const vr_request* reqs, int n_req, float* logits,
                             float* pen_logits, void* ws, size_t ws_bytes, void* stream);

/*
 * vr_verify_window with HOST inputs and outputs, for callers whose per-window
 * data lives on the host: act_h [rows][hidden], tokens_h, parent_h (or
 * NULL), q_ids_h/q_logits_h (or NULL), hist_h [hist_len] are host pointers;
 * the last min(hist_len, VR_MAX_PENALTY_WINDOW) history tokens are used.
 * weight, logits and pen_logits are device pointers.  The inputs go into ws:
 * when every input buffer is device-accessible a staging kernel reads them
 * directly, otherwise they are copied.  Device-accessible means pinned
 * (page-locked, mapped into the device's address space), or any host buffer
 * on a device that reads host memory through the host's page tables
 * (cudaDevAttrPageableMemoryAccessUsesHostPageTables, e.g. Grace systems;
 * there no buffer is queried per call).  Then the window runs; device-
 * accessible output buffers (out_ids_h [rows], and out_accept_h with
 * out_n_emitted_h) are written by the kernel, others copied back; the call
 * SYNCHRONISES the stream before returning (one wait per call).
 */
VR_API int vr_verify_window_host(const uint16_t* weight, const float* act_h, int rows, int hidden,
                          int vocab, int path, const int32_t* tokens_h, const int32_t* parent_h,
                          int n_nodes, const int32_t* q_ids_h, const float* q_logits_h,
                          const int32_t* hist_h, int hist_len, const vr_policy* policy,
                          uint64_t seed, uint64_t position, float* logits, float* pen_logits,
                          int32_t* out_ids_h, int32_t* out_accept_h, int32_t* out_n_emitted_h,
                          void* ws, size_t ws_bytes, void* stream);

/*
 * vr_verify_window_host without the wait, for a serving loop over independent
 * windows that enqueues the next window before it reads the previous one.
 * Inputs and arguments as in vr_verify_window_host.  The call stages the
 * inputs into ws as vr_verify_window_host does, enqueues the window and
 * returns.  out_h receives (2 + rows) int32: out_h[0] = accept,
 * out_h[1] = n_emitted, out_h[2 .. 2 + n_emitted) = the emitted ids (the
 * entries after them hold unspecified values).
 * Ownership and lifetime (all caller-owned):
 *   - out_h should be pinned (page-locked) host memory: the acceptance writes
 *     it directly (a pageable out_h gets one asynchronous copy); it is valid
 *     only once the stream (or an event recorded after this call) has completed;
 *   - pinned host inputs are read by the GPU after the call returns, so they
 *     must stay unchanged until the stream has passed this call;
 *   - windows enqueued on one stream with one ws run in order, each reading its
 *     own inputs.
 * Argument errors return before anything is enqueued; a device status is
 * reported as for the other calls (vr_device_status).
 */
VR_API int vr_verify_window_host_async(const uint16_t* weight, const float* act_h, int rows,
                                int hidden, int vocab, int path, const int32_t* tokens_h,
                                const int32_t* parent_h, int n_nodes, const int32_t* q_ids_h,
                                const float* q_logits_h, const int32_t* hist_h, int hist_len,
                                const vr_policy* policy, uint64_t seed, uint64_t position,
                                float* logits, float* pen_logits, int32_t* out_h, void* ws,
                                size_t ws_bytes, void* stream);

/*
 * The candidate pools of the last window (vr_verify_window, its host-buffer
 * variants or vr_verify_window_batched) enqueued with this workspace, copied
 * on `stream` into ids [rows][64] int32 and vals [rows][64] float32 (device
 * pointers, caller-owned).  Each row is the top 64 of that row's logits
 * after its penalties, in pool order ("Speculative decoding on RDNA" §03:
 * value descending, token id ascending, NaN lowest); entries past the
 * vocabulary are id -1.  For the rows of a greedy request (temperature 0)
 * only entry 0, the argmax, is defined, since that is all a greedy decision
 * uses; the other entries may be id -1.  rows, hidden and vocab are those of that call
 * (the batched call: its total rows).  Argument errors return before
 * anything is enqueued.
 */
VR_API int vr_window_pools(const void* ws, size_t ws_bytes, int rows, int hidden, int vocab,
                    int32_t* ids, float* vals, void* stream);

/* ------------------------------------------------------------------------
 * Host-side draft proposal and window pricing.  These run on the CPU, take
 * HOST pointers only, enqueue nothing and need no GPU.
 * ------------------------------------------------------------------------ */

/*
 * Prompt-lookup draft proposal ("Speculative decoding on RDNA" §06, N-gram
 * takeovers: an n-gram index of the request's whole context, by default
 * match 5 / propose 3; "One RDNA4 verify pass has slack for about two dozen
 * speculative tokens", "Spend the budget on a tree": the top few matches
 * become the branches of one token tree).
 *   1. key = the last `match` tokens of context[0..len);
 *   2. every earlier occurrence of key (start s with s + match < len)
 *      proposes context[s + match .. min(len, s + match + propose));
 *   3. identical proposals are merged and ranked by how many occurrences
 *      propose them, then by the most recent occurrence;
 *   4. the first `branches` proposals are inserted, in rank order, into one
 *      tree (a trie: a proposal sharing a prefix with an earlier one shares
 *      its nodes), new nodes appended, stopping at max_nodes nodes.
 * Out: out_tokens/out_parent [max_nodes] in the window layout above (parent
 * -1 = the root, every parent an earlier node; branches == 1 gives a chain),
 * *out_n_nodes (0 when the key has no earlier occurrence or len <= match).
 * match, propose, branches >= 1; 0 <= max_nodes <= VR_MAX_WINDOW_ROWS - 1.
 * All pointers are host memory.
 */
VR_API int vr_ngram_propose(const int32_t* context, int len, int match, int propose,
                            int branches, int max_nodes, int32_t* out_tokens,
                            int32_t* out_parent, int32_t* out_n_nodes);

/*
 * Window cost model ("Speculative decoding on RDNA" §05: window cost =
 * one-row cost + a per-row increment for each extra row).  Least-squares fit
 * of ms[i] = a + b (rows[i] - 1) over n >= 2 measured windows with at least
 * two distinct row counts.  Host pointers.
 */
VR_API int vr_cost_fit(const int32_t* rows, const double* ms, int n, double* out_a,
                       double* out_b);

/*
 * Draft depth for the next window (same page, §05): alpha[i] (in [0, 1]) is
 * the probability that draft i + 1 is accepted once drafts 1..i were;
 * E(k) = 1 + sum_{j=1..k} prod_{i<=j} alpha_i is the expected number of
 * emitted tokens with k drafts and a + b k the window's cost.  *out_k is the
 * k in [0, kmax] with the largest E(k) / (a + b k); k = 0 (one token per
 * plain step) unless a deeper window is strictly better, and the smaller k
 * among equal rates.  *out_tokens_per_ms (may be NULL) receives that rate.
 * a > 0 and a + b kmax > 0.  Host pointers.
 */
VR_API int vr_choose_depth(const double* alpha, int kmax, double a, double b, int32_t* out_k,
                           double* out_tokens_per_ms);

/*
 * N-gram takeover test (same page, §06): *out_take = 1 iff the n-gram
 * window's expected emitted tokens per unit of cost, E(alpha_ngram, k_ngram)
 * / (a + b k_ngram), is at least the native window's at its current
 * acceptance, E(alpha_native, k_native) / (a + b k_native).  k_ngram >= 1,
 * k_native >= 0.  Host pointers.
 */
VR_API int vr_takeover(const double* alpha_native, int k_native, const double* alpha_ngram,
                       int k_ngram, double a, double b, int32_t* out_take);

/*
 * The AR floor's decision (same page, §07): after one timed plain step
 * (ar_ms) and n timed probe windows (window_ms[i], emitted[i] tokens each),
 * *out_speculate = 1 iff some probe cost strictly less per emitted token
 * than the plain step.  A tie, or any invalid timing (not finite, <= 0, or a
 * probe that emitted nothing), retires the request (*out_speculate = 0).
 * Host pointers.
 */
VR_API int vr_ar_floor(double ar_ms, const double* window_ms, const int32_t* emitted, int n,
                       int32_t* out_speculate);

/*
 * Read and clear the device status word of a workspace (VR_DEV_* bits).
 * Synchronises `stream`.  Returns VR_OK, or VR_ERR_CUDA.
 */
VR_API int vr_device_status(void* ws, int32_t* out_status, void* stream);

/*
 * Zero-initialise a fresh workspace: its first 8 KiB hold the status word
 * and the ticket counters of the sampling kernel (which leaves them at zero
 * after every call).  Call once after allocating ws; enqueued on `stream`.
 */
VR_API int vr_workspace_init(void* ws, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* VERIFYROW_H */
