// C ABI of libverifyrow: argument validation, workspace layout and the
// order of launches of each entry point.  See include/verifyrow.h.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <vector>

#include "vr_common.cuh"
#include "vr_kernels.h"

namespace vr {
namespace {

constexpr size_t kAlign = 256;
// control region at the start of every workspace, zeroed by vr_workspace_init:
// the status word, then the per-row and per-request ticket counters of the
// sampling kernel (which leaves them at zero after every call)
constexpr size_t kRowTicketOff = 256;
constexpr size_t kReqTicketOff = kRowTicketOff + VR_MAX_ROWS * 4;
// then one 64-bit word per request: the done and accept bits of the rows of a
// chain (the acceptance without a walk)
constexpr size_t kReqMaskOff = kReqTicketOff + VR_MAX_REQUESTS * 4;
constexpr size_t kControlBytes = 8192;
static_assert(kReqMaskOff % 8 == 0, "control region alignment");
static_assert(kReqMaskOff + VR_MAX_REQUESTS * 8 <= kControlBytes, "control region");

struct Layout {
  size_t status, planes, cand, gmax, pool_ids, pool_vals, dec, q_pen, reqs, row_req;
  size_t st_act, st_tok, st_par, st_qid, st_qlog, st_hist, st_out, total;
};

Layout layout(int rows, int hidden, int vocab) {
  Layout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, kAlign);
    return at;
  };
  const size_t r = static_cast<size_t>(rows);
  L.status = take(kControlBytes);
  L.planes = take(std::max(tcb_plane_bytes(rows, hidden), tc_scratch_bytes(rows, hidden)));
  L.cand = take(select_cand_bytes(rows, vocab));
  L.gmax = take(r * ((static_cast<size_t>(vocab) + 31) / 32) * 4);
  L.pool_ids = take(r * kPool * 4);
  L.pool_vals = take(r * kPool * 4);
  L.dec = take(r * sizeof(int4));
  L.q_pen = take(r * kQCand * 4);
  L.reqs = take(std::min<size_t>(r, VR_MAX_REQUESTS) * sizeof(ReqDev));
  L.row_req = take(r * 4);
  L.st_act = take(r * hidden * 4);
  L.st_tok = take(r * 4);
  L.st_par = take(r * 4);
  L.st_qid = take(r * kQCand * 4);
  L.st_qlog = take(r * kQCand * 4);
  L.st_hist = take(VR_MAX_PENALTY_WINDOW * 4);
  L.st_out = take((r + 2) * 4);
  L.total = off;
  return L;
}

template <class T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

bool finite(float x) { return std::isfinite(x); }

int check_policy(const vr_policy* p) {
  if (!p) return VR_ERR_ARG;
  if (!finite(p->temperature) || p->temperature < 0.f) return VR_ERR_ARG;
  if (!finite(p->min_p) || !finite(p->top_p)) return VR_ERR_ARG;
  if (!finite(p->repeat) || p->repeat <= 0.f) return VR_ERR_ARG;
  if (!finite(p->presence) || !finite(p->frequency)) return VR_ERR_ARG;
  if (p->window < 0 || p->window > VR_MAX_PENALTY_WINDOW) return VR_ERR_ARG;
  return VR_OK;
}

bool active(const vr_policy& p) {
  return p.window > 0 && (p.repeat != 1.f || p.presence != 0.f || p.frequency != 0.f);
}

int check_shape(int rows, int hidden, int vocab) {
  if (rows < 1 || rows > VR_MAX_ROWS) return VR_ERR_ARG;
  if (vocab < 1) return VR_ERR_ARG;
  if (hidden < 8 || hidden > 65536) return VR_ERR_ARG;
  if (hidden % 8) return VR_ERR_UNSUPPORTED;
  return VR_OK;
}

int check_ws(void* ws, size_t ws_bytes, int rows, int hidden, int vocab) {
  if (!ws || reinterpret_cast<uintptr_t>(ws) % kAlign) return VR_ERR_WORKSPACE;
  if (ws_bytes < layout(rows, hidden, vocab).total) return VR_ERR_WORKSPACE;
  return VR_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_window(int rows, int n_nodes, const int32_t* tokens, const int32_t* q_ids,
                 const float* q_logits, const int32_t* hist, int hist_len) {
  if (n_nodes < 0 || rows != n_nodes + 1 || rows > VR_MAX_WINDOW_ROWS) return VR_ERR_ARG;
  if (n_nodes > 0 && !tokens) return VR_ERR_ARG;
  if ((q_ids == nullptr) != (q_logits == nullptr)) return VR_ERR_ARG;
  if (hist_len < 0 || (hist_len > 0 && !hist)) return VR_ERR_ARG;
  return VR_OK;
}

ReqDev make_req(int row0, int n_nodes, const int32_t* tokens, const int32_t* parent,
                const int32_t* q_ids, const float* q_in, float* q_pen, const int32_t* hist,
                int hist_len, const vr_policy& pol, uint64_t seed, uint64_t position,
                int32_t* out_ids, int32_t* out_accept, int32_t* out_n) {
  ReqDev r{};
  r.row0 = row0;
  r.n_nodes = n_nodes;
  r.tokens = tokens;
  r.parent = parent;
  r.q_ids = q_ids;
  r.q_logits_in = q_in;
  r.q_pen = q_pen;
  r.hist = hist;
  r.hist_len = hist_len;
  r.pol = pol;
  r.seed = seed;
  r.position = position;
  r.out_ids = out_ids;
  r.out_accept = out_accept;
  r.out_n = out_n;
  return r;
}

ReqTable single(const ReqDev& r) {
  ReqTable t{};
  t.one = r;
  t.many = nullptr;
  t.row_req = nullptr;
  t.n_req = 1;
  return t;
}


// gmax (nullable): where the tensor-core paths also record the group maxima
// logits2 (nullable): a second buffer receiving the same logits (the
// tensor-core epilogues write both; the CUDA-core path copies)
int project(const uint16_t* weight, const float* act, int rows, int hidden, int vocab, int path,
            float* logits, float* logits2, uint32_t* gmax, void* ws, const Layout& L,
            cudaStream_t s) {
  if (path == VR_PATH_AUTO) path = VR_PATH_TC;
  if (path == VR_PATH_TC)
    return launch_project_tc(weight, act, rows, hidden, vocab, logits, logits2,
                             at<void>(ws, L.planes), gmax, at<int32_t>(ws, L.status), s);
  if (path == VR_PATH_TC_BATCH)
    return launch_project_tcb(weight, act, rows, hidden, vocab, logits, logits2,
                              at<void>(ws, L.planes), gmax, at<int32_t>(ws, L.status), s);
  if (path == VR_PATH_FFMA) {
    const int st = launch_project_ffma(weight, act, rows, hidden, vocab, logits, s);
    if (st != VR_OK || !logits2) return st;
    return cudaMemcpyAsync(logits2, logits, static_cast<size_t>(rows) * vocab * sizeof(float),
                           cudaMemcpyDeviceToDevice, s) == cudaSuccess
               ? VR_OK
               : VR_ERR_CUDA;
  }
  return VR_ERR_ARG;
}

// True when the projection path records group maxima for the sampling stage
bool records_gmax(int path, int vocab) {
  return (path == VR_PATH_AUTO || path == VR_PATH_TC || path == VR_PATH_TC_BATCH) &&
         sample_rows_supported(vocab);
}

// True when the row sampling kernel after a projection on `path` starts well
// before its wait returns: its CTAs, two per SM, fit on the SMs that the
// tensor-core projection leaves free from its start or frees a unit of work
// before its end.  It may then warm its instruction cache before the wait.
bool row_kernel_starts_early(int path, int rows, int vocab) {
  if (path != VR_PATH_AUTO && path != VR_PATH_TC) return false;
  return (rows + 1) / 2 <= tc_early_free_sms(rows, vocab);
}

// penalties -> pool + policy -> acceptance, for requests already in `tab`;
// gmax: the group maxima of `target` if the projection recorded them; early:
// row_kernel_starts_early for the projection that ran
int sample_stages(const ReqTable& tab, int n_req, int rows, int vocab, float* target,
                  uint32_t* gmax, bool any_active, bool any_q, bool early, void* ws,
                  const Layout& L, cudaStream_t s) {
  (void)n_req;
  // windows on a tensor-core path: the row kernel applies the penalties itself
  if (gmax)
    return launch_sample_rows(target, rows, vocab, gmax, at<uint32_t>(ws, L.status + kReqTicketOff),
                              at<unsigned long long>(ws, L.status + kReqMaskOff),
                              at<int32_t>(ws, L.pool_ids), at<float>(ws, L.pool_vals), tab,
                              at<int4>(ws, L.dec), at<int32_t>(ws, L.status),
                              any_active ? target : nullptr, early, s);
  int st;
  if (any_active) {
    st = launch_penalize(tab, rows, target, vocab, any_q, at<int32_t>(ws, L.status), s);
    if (st != VR_OK) return st;
  }
  return launch_sample(target, rows, vocab, at<uint64_t>(ws, L.cand),
                       at<uint32_t>(ws, L.status + kRowTicketOff),
                       at<uint32_t>(ws, L.status + kReqTicketOff),
                       at<unsigned long long>(ws, L.status + kReqMaskOff), at<int32_t>(ws, L.pool_ids),
                       at<float>(ws, L.pool_vals), &tab, at<int4>(ws, L.dec),
                       at<int32_t>(ws, L.status), s);
}

int window_device(const uint16_t* weight, const float* act, int rows, int hidden, int vocab,
                  int path, const int32_t* tokens, const int32_t* parent, int n_nodes,
                  const int32_t* q_ids, const float* q_logits, const int32_t* hist, int hist_len,
                  const vr_policy& pol, uint64_t seed, uint64_t position, float* logits,
                  float* pen_logits, int32_t* out_ids, int32_t* out_accept, int32_t* out_n,
                  void* ws, const Layout& L, cudaStream_t s) {
  uint32_t* gmax = records_gmax(path, vocab) ? at<uint32_t>(ws, L.gmax) : nullptr;
  const bool act_pen = active(pol);
  // penalties into a separate buffer: the projection writes both copies
  float* target = (act_pen && pen_logits) ? pen_logits : logits;
  int st = project(weight, act, rows, hidden, vocab, path, logits,
                   target != logits ? target : nullptr, gmax, ws, L, s);
  if (st != VR_OK) return st;
  float* q_pen = (act_pen && q_ids) ? at<float>(ws, L.q_pen) : const_cast<float*>(q_logits);
  const ReqTable tab = single(make_req(0, n_nodes, tokens, parent, q_ids, q_logits, q_pen, hist,
                                       hist_len, pol, seed, position, out_ids, out_accept, out_n));
  return sample_stages(tab, 1, rows, vocab, target, gmax, act_pen, q_ids != nullptr,
                       row_kernel_starts_early(path, rows, vocab), ws, L, s);
}

}  // namespace
}  // namespace vr

using namespace vr;

extern "C" {

int vr_abi_version(void) { return VR_ABI_VERSION; }

const char* vr_status_string(int status) {
  switch (status) {
    case VR_OK: return "ok";
    case VR_ERR_ARG: return "invalid argument";
    case VR_ERR_CUDA: return "CUDA error";
    case VR_ERR_UNSUPPORTED: return "unsupported shape";
    case VR_ERR_DEVICE: return "device status word set";
    case VR_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    default: return "unknown status";
  }
}

int vr_workspace_bytes(int rows, int hidden, int vocab, size_t* out_bytes) {
  if (!out_bytes) return VR_ERR_ARG;
  const int st = check_shape(rows, hidden, vocab);
  if (st != VR_OK) return st;
  *out_bytes = layout(rows, hidden, vocab).total;
  return VR_OK;
}

int vr_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || ws_bytes < kControlBytes || reinterpret_cast<uintptr_t>(ws) % kAlign)
    return VR_ERR_WORKSPACE;
  return cudaMemsetAsync(ws, 0, kControlBytes, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? VR_OK
             : VR_ERR_CUDA;
}

int vr_verify_project(const uint16_t* weight, const float* act, int rows, int hidden, int vocab,
                      int path, float* logits, void* ws, size_t ws_bytes, void* stream) {
  int st = check_shape(rows, hidden, vocab);
  if (st != VR_OK) return st;
  if (!weight || !act || !logits) return VR_ERR_ARG;
  if (path < VR_PATH_AUTO || path > VR_PATH_TC_BATCH) return VR_ERR_ARG;
  if (!aligned16(weight)) return VR_ERR_ARG;
  if ((st = check_ws(ws, ws_bytes, rows, hidden, vocab)) != VR_OK) return st;
  return project(weight, act, rows, hidden, vocab, path, logits, nullptr, nullptr, ws,
                 layout(rows, hidden, vocab), static_cast<cudaStream_t>(stream));
}

int vr_verify_penalize(float* logits, int rows, int vocab, const int32_t* tokens,
                       const int32_t* parent, int n_nodes, const int32_t* hist, int hist_len,
                       const vr_policy* policy, const int32_t* q_ids, float* q_logits, void* ws,
                       size_t ws_bytes, void* stream) {
  int st = check_policy(policy);
  if (st != VR_OK) return st;
  if (!logits || vocab < 1) return VR_ERR_ARG;
  if ((st = check_window(rows, n_nodes, tokens, q_ids, q_logits, hist, hist_len)) != VR_OK) return st;
  if ((st = check_ws(ws, ws_bytes, rows, 8, vocab)) != VR_OK) return st;
  if (!active(*policy)) return VR_OK;
  const ReqTable tab = single(make_req(0, n_nodes, tokens, parent, q_ids, q_logits, q_logits, hist,
                                       hist_len, *policy, 0, 0, nullptr, nullptr, nullptr));
  const Layout L = layout(rows, 8, vocab);
  return launch_penalize(tab, rows, logits, vocab, q_ids != nullptr,
                         at<int32_t>(ws, L.status), static_cast<cudaStream_t>(stream));
}

int vr_verify_select(const float* logits, int rows, int vocab, int32_t* pool_ids,
                     float* pool_vals, void* ws, size_t ws_bytes, void* stream) {
  int st = check_shape(rows, 8, vocab);
  if (st != VR_OK) return st;
  if (!logits || !pool_ids || !pool_vals) return VR_ERR_ARG;
  if ((st = check_ws(ws, ws_bytes, rows, 8, vocab)) != VR_OK) return st;
  const Layout L = layout(rows, 8, vocab);
  return launch_sample(logits, rows, vocab, at<uint64_t>(ws, L.cand),
                       at<uint32_t>(ws, L.status + kRowTicketOff),
                       at<uint32_t>(ws, L.status + kReqTicketOff), nullptr, pool_ids, pool_vals,
                       nullptr,
                       nullptr, at<int32_t>(ws, L.status), static_cast<cudaStream_t>(stream));
}

int vr_topk(const float* x, int rows, int vocab, int k, int32_t* ids, float* vals, void* ws,
            size_t ws_bytes, void* stream) {
  int st = check_shape(rows, 8, vocab);
  if (st != VR_OK) return st;
  if (!x || !ids || !vals || k < 1 || k > VR_POOL) return VR_ERR_ARG;
  if ((st = check_ws(ws, ws_bytes, rows, 8, vocab)) != VR_OK) return st;
  const Layout L = layout(rows, 8, vocab);
  return launch_sample(x, rows, vocab, at<uint64_t>(ws, L.cand),
                       at<uint32_t>(ws, L.status + kRowTicketOff),
                       at<uint32_t>(ws, L.status + kReqTicketOff), nullptr, ids, vals, nullptr,
                       nullptr,
                       at<int32_t>(ws, L.status), static_cast<cudaStream_t>(stream), k);
}

int vr_verify_policy(const float* pool_vals, int rows, int pool_len, const vr_policy* policy,
                     int32_t* out_m, float* out_e, float* out_S, void* stream) {
  int st = check_policy(policy);
  if (st != VR_OK) return st;
  if (!pool_vals || !out_m || !out_e || !out_S) return VR_ERR_ARG;
  if (rows < 1 || rows > VR_MAX_ROWS || pool_len < 1 || pool_len > VR_POOL) return VR_ERR_ARG;
  return launch_policy(pool_vals, rows, pool_len, *policy, out_m, out_e, out_S,
                       static_cast<cudaStream_t>(stream));
}

int vr_verify_sample_accept(const float* pen_logits, int rows, int vocab, const int32_t* tokens,
                            const int32_t* parent, int n_nodes, const int32_t* q_ids,
                            const float* q_logits, const vr_policy* policy, uint64_t seed,
                            uint64_t position, int32_t* out_ids, int32_t* out_accept,
                            int32_t* out_n_emitted, void* ws, size_t ws_bytes, void* stream) {
  int st = check_policy(policy);
  if (st != VR_OK) return st;
  if (!pen_logits || vocab < 1 || !out_ids || !out_accept || !out_n_emitted) return VR_ERR_ARG;
  if ((st = check_window(rows, n_nodes, tokens, q_ids, q_logits, nullptr, 0)) != VR_OK) return st;
  if ((st = check_ws(ws, ws_bytes, rows, 8, vocab)) != VR_OK) return st;
  const Layout L = layout(rows, 8, vocab);
  const ReqTable tab =
      single(make_req(0, n_nodes, tokens, parent, q_ids, q_logits, const_cast<float*>(q_logits),
                      nullptr, 0, *policy, seed, position, out_ids, out_accept, out_n_emitted));
  return sample_stages(tab, 1, rows, vocab, const_cast<float*>(pen_logits), nullptr, false, false,
                       false, ws, L, static_cast<cudaStream_t>(stream));
}

int vr_verify_window(const uint16_t* weight, const float* act, int rows, int hidden, int vocab,
                     int path, const int32_t* tokens, const int32_t* parent, int n_nodes,
                     const int32_t* q_ids, const float* q_logits, const int32_t* hist,
                     int hist_len, const vr_policy* policy, uint64_t seed, uint64_t position,
                     float* logits, float* pen_logits, int32_t* out_ids, int32_t* out_accept,
                     int32_t* out_n_emitted, void* ws, size_t ws_bytes, void* stream) {
  int st = check_policy(policy);
  if (st != VR_OK) return st;
  if ((st = check_shape(rows, hidden, vocab)) != VR_OK) return st;
  if (!weight || !act || !logits || !out_ids || !out_accept || !out_n_emitted) return VR_ERR_ARG;
  if (path < VR_PATH_AUTO || path > VR_PATH_TC_BATCH || !aligned16(weight)) return VR_ERR_ARG;
  if ((st = check_window(rows, n_nodes, tokens, q_ids, q_logits, hist, hist_len)) != VR_OK) return st;
  if ((st = check_ws(ws, ws_bytes, rows, hidden, vocab)) != VR_OK) return st;
  return window_device(weight, act, rows, hidden, vocab, path, tokens, parent, n_nodes, q_ids,
                       q_logits, hist, hist_len, *policy, seed, position, logits, pen_logits,
                       out_ids, out_accept, out_n_emitted, ws, layout(rows, hidden, vocab),
                       static_cast<cudaStream_t>(stream));
}

int vr_verify_window_batched(const uint16_t* weight, const float* act, int hidden, int vocab,
                             int path, const vr_request* reqs, int n_req, float* logits,
                             float* pen_logits, void* ws, size_t ws_bytes, void* stream) {
  if (!reqs || n_req < 1 || n_req > VR_MAX_REQUESTS) return VR_ERR_ARG;
  if (!weight || !act || !logits || !aligned16(weight)) return VR_ERR_ARG;
  if (path < VR_PATH_AUTO || path > VR_PATH_TC_BATCH) return VR_ERR_ARG;
  int rows = 0, st;
  bool any_active = false, any_q = false;
  for (int b = 0; b < n_req; ++b) {
    const vr_request& r = reqs[b];
    if ((st = check_policy(&r.policy)) != VR_OK) return st;
    if ((st = check_window(r.n_nodes + 1, r.n_nodes, r.tokens, r.q_ids, r.q_logits, r.hist,
                           r.hist_len)) != VR_OK)
      return st;
    if (!r.out_ids || !r.out_accept || !r.out_n_emitted) return VR_ERR_ARG;
    rows += r.n_nodes + 1;
    if (rows > VR_MAX_ROWS) return VR_ERR_ARG;
    any_active |= active(r.policy);
    any_q |= r.q_ids != nullptr;
  }
  if ((st = check_shape(rows, hidden, vocab)) != VR_OK) return st;
  if ((st = check_ws(ws, ws_bytes, rows, hidden, vocab)) != VR_OK) return st;
  const Layout L = layout(rows, hidden, vocab);
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  std::vector<ReqDev> table(n_req);
  int row0 = 0;
  for (int b = 0; b < n_req; ++b) {
    const vr_request& r = reqs[b];
    float* q_pen = (active(r.policy) && r.q_ids) ? at<float>(ws, L.q_pen) + static_cast<size_t>(row0) * kQCand
                                                : const_cast<float*>(r.q_logits);
    table[b] = make_req(row0, r.n_nodes, r.tokens, r.parent, r.q_ids, r.q_logits, q_pen, r.hist,
                        r.hist_len, r.policy, r.seed, r.position, r.out_ids, r.out_accept,
                        r.out_n_emitted);
    row0 += r.n_nodes + 1;
  }
  // staged by kernels that carry the table in their parameters (copied at
  // launch or capture): no operation on the stream reads this call's host
  // memory, so the call can be captured into a graph and replayed
  if ((st = launch_stage_requests(table.data(), n_req, at<ReqDev>(ws, L.reqs),
                                  at<int32_t>(ws, L.row_req), s)) != VR_OK)
    return st;

  uint32_t* gmax = records_gmax(path, vocab) ? at<uint32_t>(ws, L.gmax) : nullptr;
  // penalties into a separate buffer: the projection writes both copies
  float* target = (any_active && pen_logits) ? pen_logits : logits;
  st = project(weight, act, rows, hidden, vocab, path, logits, target != logits ? target : nullptr,
               gmax, ws, L, s);
  if (st != VR_OK) return st;
  ReqTable tab{};
  tab.many = at<ReqDev>(ws, L.reqs);
  tab.row_req = at<int32_t>(ws, L.row_req);
  tab.n_req = n_req;
  return sample_stages(tab, n_req, rows, vocab, target, gmax, any_active, any_q,
                       row_kernel_starts_early(path, rows, vocab), ws, L, s);
}

}  // extern "C"

namespace {

// True when kernels on the current device can read and write any host
// address through the host's page tables (a coherent CPU-GPU system such as
// Grace with ATS): then every host buffer is device-accessible at its own
// address, pinned or not.  Looked up once per device.
bool host_pages_device_visible() {
  static std::atomic<int> state[kMaxDevices];     // 0 unknown, 1 no, 2 yes
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  const bool cached = dev >= 0 && dev < kMaxDevices;
  if (cached) {
    const int v = state[dev].load(std::memory_order_acquire);
    if (v) return v == 2;
  }
  int attr = 0;
  const bool yes = cudaDeviceGetAttribute(&attr, cudaDevAttrPageableMemoryAccessUsesHostPageTables,
                                          dev) == cudaSuccess &&
                   attr != 0;
  if (!yes) cudaGetLastError();
  if (cached) state[dev].store(yes ? 2 : 1, std::memory_order_release);
  return yes;
}

// The device address of a host buffer that kernels may read and write: with
// `direct` (the caller waits for the window before returning, and host pages
// are device-visible) the buffer itself, with no driver query per call;
// else the mapping of a pinned (page-locked, device-mapped) buffer, or
// nullptr when the buffer is pageable (then it is copied instead).
template <class T>
T* mapped(T* p, bool direct = false) {
  if (!p) return nullptr;
  if (direct) return p;
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost || !a.devicePointer) return nullptr;
  return static_cast<T*>(a.devicePointer);
}

// The host-buffer window: checks, the inputs into ws (read by the staging
// kernel from pinned memory, else copied), then the window itself, whose
// acceptance writes ids/accept/n to the given device-writable addresses.
int window_host_enqueue(const uint16_t* weight, const float* act_h, int rows, int hidden,
                        int vocab, int path, const int32_t* tokens_h, const int32_t* parent_h,
                        int n_nodes, const int32_t* q_ids_h, const float* q_logits_h,
                        const int32_t* hist_h, int hist_len, const vr_policy* policy,
                        uint64_t seed, uint64_t position, float* logits, float* pen_logits,
                        void* ws, size_t ws_bytes, cudaStream_t s, int32_t* ids_dst,
                        int32_t* accept_dst, int32_t* n_dst, bool direct) {
  const Layout L = layout(rows, hidden, vocab);
  const int h_keep = std::min(hist_len, VR_MAX_PENALTY_WINDOW);
  const int32_t* hist_tail = h_keep > 0 ? hist_h + (hist_len - h_keep) : nullptr;
  struct In {
    const void* h;
    size_t off, words;
  };
  const In in[kMaxStageSegs] = {
      {act_h, L.st_act, static_cast<size_t>(rows) * hidden},
      {n_nodes ? tokens_h : nullptr, L.st_tok, static_cast<size_t>(n_nodes)},
      {parent_h, L.st_par, static_cast<size_t>(n_nodes)},
      {q_ids_h, L.st_qid, static_cast<size_t>(n_nodes) * kQCand},
      {q_logits_h, L.st_qlog, static_cast<size_t>(n_nodes) * kQCand},
      {hist_tail, L.st_hist, static_cast<size_t>(h_keep)}};
  StageSeg seg[kMaxStageSegs];
  int nseg = 0;
  bool all_mapped = true;
  for (const In& x : in) {
    if (!x.h || x.words == 0) continue;
    const void* m = mapped(x.h, direct);
    if (!m) {
      all_mapped = false;
      break;
    }
    seg[nseg++] = {static_cast<const uint32_t*>(m), at<uint32_t>(ws, x.off),
                   static_cast<uint32_t>(x.words)};
  }
  if (all_mapped) {
    const int st = launch_stage_inputs(seg, nseg, s);
    if (st != VR_OK) return st;
  } else {
    for (const In& x : in)
      if (x.h && x.words &&
          cudaMemcpyAsync(at<void>(ws, x.off), x.h, x.words * 4, cudaMemcpyHostToDevice, s) !=
              cudaSuccess)
        return VR_ERR_CUDA;
  }
  return window_device(weight, at<float>(ws, L.st_act), rows, hidden, vocab, path,
                       at<int32_t>(ws, L.st_tok), parent_h ? at<int32_t>(ws, L.st_par) : nullptr,
                       n_nodes, q_ids_h ? at<int32_t>(ws, L.st_qid) : nullptr,
                       q_logits_h ? at<float>(ws, L.st_qlog) : nullptr, at<int32_t>(ws, L.st_hist),
                       h_keep, *policy, seed, position, logits, pen_logits, ids_dst, accept_dst,
                       n_dst, ws, L, s);
}

int check_host_window(const uint16_t* weight, const float* act_h, int rows, int hidden, int vocab,
                      int path, const int32_t* tokens_h, int n_nodes, const int32_t* q_ids_h,
                      const float* q_logits_h, const int32_t* hist_h, int hist_len,
                      const vr_policy* policy, const float* logits, void* ws, size_t ws_bytes) {
  int st = check_policy(policy);
  if (st != VR_OK) return st;
  if ((st = check_shape(rows, hidden, vocab)) != VR_OK) return st;
  if (!weight || !act_h || !logits) return VR_ERR_ARG;
  if (path < VR_PATH_AUTO || path > VR_PATH_TC_BATCH || !aligned16(weight)) return VR_ERR_ARG;
  if ((st = check_window(rows, n_nodes, tokens_h, q_ids_h, q_logits_h, hist_h, hist_len)) != VR_OK)
    return st;
  return check_ws(ws, ws_bytes, rows, hidden, vocab);
}

}  // namespace

extern "C" {

int vr_verify_window_host(const uint16_t* weight, const float* act_h, int rows, int hidden,
                          int vocab, int path, const int32_t* tokens_h, const int32_t* parent_h,
                          int n_nodes, const int32_t* q_ids_h, const float* q_logits_h,
                          const int32_t* hist_h, int hist_len, const vr_policy* policy,
                          uint64_t seed, uint64_t position, float* logits, float* pen_logits,
                          int32_t* out_ids_h, int32_t* out_accept_h, int32_t* out_n_emitted_h,
                          void* ws, size_t ws_bytes, void* stream) {
  if (!out_ids_h || !out_accept_h || !out_n_emitted_h) return VR_ERR_ARG;
  int st = check_host_window(weight, act_h, rows, hidden, vocab, path, tokens_h, n_nodes, q_ids_h,
                             q_logits_h, hist_h, hist_len, policy, logits, ws, ws_bytes);
  if (st != VR_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* out = at<int32_t>(ws, layout(rows, hidden, vocab).st_out);
  // pinned output buffers are written by the acceptance kernel; the others
  // are staged in ws and copied
  // the call waits for the window, so where host pages are device-visible
  // every host buffer is used at its own address (no copies, no queries)
  const bool direct = host_pages_device_visible();
  int32_t* ids_dev = mapped(out_ids_h, direct);
  int32_t* acc_dev = mapped(out_accept_h, direct);
  int32_t* n_dev = mapped(out_n_emitted_h, direct);
  const bool head_dev = acc_dev && n_dev;
  st = window_host_enqueue(weight, act_h, rows, hidden, vocab, path, tokens_h, parent_h, n_nodes,
                           q_ids_h, q_logits_h, hist_h, hist_len, policy, seed, position, logits,
                           pen_logits, ws, ws_bytes, s, ids_dev ? ids_dev : out + 2,
                           head_dev ? acc_dev : out, head_dev ? n_dev : out + 1, direct);
  if (st != VR_OK) return st;
  // a pageable accept/n copy is the last one enqueued: the call waits once
  int32_t head[2];
  if ((!ids_dev && cudaMemcpyAsync(out_ids_h, out + 2, static_cast<size_t>(rows) * sizeof(int32_t),
                                   cudaMemcpyDeviceToHost, s) != cudaSuccess) ||
      (!head_dev &&
       cudaMemcpyAsync(head, out, 2 * sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess) ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return VR_ERR_CUDA;
  if (!head_dev) {
    *out_accept_h = head[0];
    *out_n_emitted_h = head[1];
  }
  return VR_OK;
}

int vr_verify_window_host_async(const uint16_t* weight, const float* act_h, int rows, int hidden,
                                int vocab, int path, const int32_t* tokens_h,
                                const int32_t* parent_h, int n_nodes, const int32_t* q_ids_h,
                                const float* q_logits_h, const int32_t* hist_h, int hist_len,
                                const vr_policy* policy, uint64_t seed, uint64_t position,
                                float* logits, float* pen_logits, int32_t* out_h, void* ws,
                                size_t ws_bytes, void* stream) {
  if (!out_h) return VR_ERR_ARG;
  int st = check_host_window(weight, act_h, rows, hidden, vocab, path, tokens_h, n_nodes, q_ids_h,
                             q_logits_h, hist_h, hist_len, policy, logits, ws, ws_bytes);
  if (st != VR_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // pinned out_h: the acceptance writes it directly; otherwise one copy
  int32_t* dev = mapped(out_h);
  int32_t* out = dev ? dev : at<int32_t>(ws, layout(rows, hidden, vocab).st_out);
  st = window_host_enqueue(weight, act_h, rows, hidden, vocab, path, tokens_h, parent_h, n_nodes,
                           q_ids_h, q_logits_h, hist_h, hist_len, policy, seed, position, logits,
                           pen_logits, ws, ws_bytes, s, out + 2, out, out + 1, false);
  if (st != VR_OK || dev) return st;
  return cudaMemcpyAsync(out_h, out, static_cast<size_t>(2 + rows) * sizeof(int32_t),
                         cudaMemcpyDeviceToHost, s) == cudaSuccess
             ? VR_OK
             : VR_ERR_CUDA;
}

int vr_window_pools(const void* ws, size_t ws_bytes, int rows, int hidden, int vocab, int32_t* ids,
                    float* vals, void* stream) {
  if (!ids || !vals) return VR_ERR_ARG;
  int st = check_shape(rows, hidden, vocab);
  if (st != VR_OK) return st;
  if ((st = check_ws(const_cast<void*>(ws), ws_bytes, rows, hidden, vocab)) != VR_OK) return st;
  const Layout L = layout(rows, hidden, vocab);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t bytes = static_cast<size_t>(rows) * kPool * 4;
  void* w = const_cast<void*>(ws);
  return cudaMemcpyAsync(ids, at<int32_t>(w, L.pool_ids), bytes, cudaMemcpyDeviceToDevice, s) ==
                     cudaSuccess &&
                 cudaMemcpyAsync(vals, at<float>(w, L.pool_vals), bytes, cudaMemcpyDeviceToDevice,
                                 s) == cudaSuccess
             ? VR_OK
             : VR_ERR_CUDA;
}

int vr_device_status(void* ws, int32_t* out_status, void* stream) {
  if (!ws || !out_status) return VR_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, ws, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemsetAsync(ws, 0, sizeof(int32_t), s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return VR_ERR_CUDA;
  *out_status = v;
  return VR_OK;
}

}  // extern "C"
