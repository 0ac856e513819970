// Device-side building blocks shared by the verifyrow kernels.
//
// Every floating-point step that decides an integer (a pool order, a kept
// count, a draw) uses explicit round-to-nearest intrinsics, so that no
// fused multiply-add or fast-math rewrite can change a bit; the library is
// also compiled with --fmad=false.  The sampler works in float32 (the pages
// fix no precision; GB300's double-precision latency made the per-row
// decisions a tenth of the window).
#pragma once

#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

#include "../../include/verifyrow.h"

namespace vr {

constexpr int kPool = VR_POOL;
constexpr int kQCand = VR_QCAND;
constexpr int kTopKAbsent = 20;

// ---------------------------------------------------------------------------
// status word (first int32 of the workspace)

__device__ __forceinline__ void set_status(int32_t* status, int32_t bits) {
  if (status) atomicOr(reinterpret_cast<int*>(status), bits);
}

// ---------------------------------------------------------------------------
// request table.  A single-window call passes its one request by value; a
// batched call passes a device array.

struct ReqDev {
  int32_t row0;         // first row of the request in the stacked rows
  int32_t n_nodes;      // rows of the request = n_nodes + 1
  const int32_t* tokens;
  const int32_t* parent;     // nullptr = chain
  const int32_t* q_ids;      // nullptr = no draft candidates
  const float* q_logits_in;  // candidates' logits as given
  float* q_pen;              // [n_nodes][8] penalised copy (workspace) or in place
  const int32_t* hist;
  int32_t hist_len;
  vr_policy pol;
  uint64_t seed;
  uint64_t position;
  int32_t* out_ids;
  int32_t* out_accept;
  int32_t* out_n;
};

struct ReqTable {
  ReqDev one;
  const ReqDev* many;        // nullptr => `one` is the only request
  const int32_t* row_req;    // [rows] request of each row (batched only)
  int32_t n_req;
};

__device__ __forceinline__ const ReqDev& request(const ReqTable& t, int b) {
  return t.many ? t.many[b] : t.one;
}
__device__ __forceinline__ int request_of_row(const ReqTable& t, int row) {
  return t.many ? t.row_req[row] : 0;
}

__device__ __forceinline__ bool penalties_active(const vr_policy& p) {
  return p.window > 0 && (p.repeat != 1.f || p.presence != 0.f || p.frequency != 0.f);
}

// ---------------------------------------------------------------------------
// total order of float32 used by the pool: unsigned order of the key below
// is value order with every NaN lowest and -0.0 below +0.0.

// Loads of data a preceding kernel of the same window wrote (logits, group
// maxima).  With programmatic dependent launch a kernel can be resident
// before its predecessor finishes, so these go through L2 only (.cg), never
// through a possibly stale L1 line.  ld_logit is volatile: issued where
// written and its value held in a register, never dropped and re-read later
// under register pressure.
__device__ __forceinline__ float ld_logit(const float* p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t float_key(float x) {
  const uint32_t b = __float_as_uint(x);
  if (isnan(x)) return 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// (key, id) packed so that a larger value means earlier in pool order:
// key descending, then id ascending.  id < 2^31, so the low word is > 0 and
// a packed value of 0 never names a real entry.
__device__ __forceinline__ uint64_t pack_key_id(uint32_t key, uint32_t id) {
  return (static_cast<uint64_t>(key) << 32) | static_cast<uint64_t>(~id);
}
__device__ __forceinline__ uint32_t packed_id(uint64_t p) {
  return ~static_cast<uint32_t>(p & 0xFFFFFFFFull);
}

// ---------------------------------------------------------------------------
// Philox4x64-10 (Salmon et al., SC'11): counter (position, row, purpose, 0),
// key (seed, 0); u = (word0 >> 40) * 2^-24, a float32 in [0, 1).

constexpr uint64_t kPhiloxM0 = 0xD2E7470EE14C6C93ull;
constexpr uint64_t kPhiloxM1 = 0xCA5A826395121157ull;
constexpr uint64_t kPhiloxW0 = 0x9E3779B97F4A7C15ull;
constexpr uint64_t kPhiloxW1 = 0xBB67AE8584CAA73Bull;
constexpr int kPurposeAccept = 1;
constexpr int kPurposeEmit = 2;

__device__ __forceinline__ uint64_t philox_word0(uint64_t c0, uint64_t c1, uint64_t c2,
                                                 uint64_t c3, uint64_t k0, uint64_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += kPhiloxW0;
      k1 += kPhiloxW1;
    }
    const uint64_t lo0 = kPhiloxM0 * c0, hi0 = __umul64hi(kPhiloxM0, c0);
    const uint64_t lo1 = kPhiloxM1 * c2, hi1 = __umul64hi(kPhiloxM1, c2);
    const uint64_t n0 = hi1 ^ c1 ^ k0;
    const uint64_t n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
  }
  return c0;
}

__device__ __forceinline__ float uniform01(uint64_t seed, uint64_t position, uint64_t row,
                                           uint64_t purpose) {
  const uint64_t w = philox_word0(position, row, purpose, 0ull, seed, 0ull);
  return __fmul_rn(__uint2float_rn(static_cast<uint32_t>(w >> 40)), 0x1p-24f);
}

// ---------------------------------------------------------------------------
// vexp: Cody-Waite reduction by ln 2 (C1 = ln 2 in float32 with its low 8
// significand bits cleared, C2 = nearest float32 to ln 2 - C1), degree-7
// Taylor polynomial of e^r in Horner form (coefficients: the float32 nearest
// to 1/j!), scaling by 2^n from the exponent bits.  float32 +, -, x only,
// each rounded to nearest; 0 below -87, so every result is normal.

__device__ __forceinline__ float vexp(float z) {
  if (!(z >= -87.0f)) return 0.0f;
  if (z > 88.0f) return __int_as_float(0x7f800000);
  const float kInvLn2 = __int_as_float(0x3fb8aa3b);
  const float kC1 = __int_as_float(0x3f317200);
  const float kC2 = __int_as_float(0x35bfbe8e);
  const float nf = rintf(__fmul_rn(z, kInvLn2));
  const float r = __fsub_rn(__fsub_rn(z, __fmul_rn(nf, kC1)), __fmul_rn(nf, kC2));
  float p = __int_as_float(0x39500d01);                       // 1/7!
  p = __fadd_rn(__fmul_rn(p, r), __int_as_float(0x3ab60b61));  // 1/6!
  p = __fadd_rn(__fmul_rn(p, r), __int_as_float(0x3c088889));  // 1/5!
  p = __fadd_rn(__fmul_rn(p, r), __int_as_float(0x3d2aaaab));  // 1/4!
  p = __fadd_rn(__fmul_rn(p, r), __int_as_float(0x3e2aaaab));  // 1/3!
  p = __fadd_rn(__fmul_rn(p, r), 0.5f);                        // 1/2!
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);                        // 1/1!
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);                        // 1/0!
  const int n = static_cast<int>(nf);
  return __fmul_rn(p, __int_as_float((n + 127) << 23));
}

// A block barrier that every warp reaches as a whole.  __syncthreads counts
// arrivals per warp, so lanes that branched apart just before (one lane
// walking a loop while the others skip it) must reconverge first; a barrier
// reached by a warp in pieces can release before the late lanes arrive.
__device__ __forceinline__ void block_sync() {
  __syncwarp();
  __syncthreads();
}

// ---------------------------------------------------------------------------
// penalty history ("Speculative decoding on RDNA" §04): H[0..len) = the last
// W = pol.window tokens of (hist || tokens on the path root -> end_node),
// end_node = -1 for the request's root row.  The path follows the parent
// array (NULL: a chain).  All NT threads of the CTA call it: they stage the
// parents in shared memory, one thread walks them there, and all copy the
// history and the path's tokens (the loads overlap).  par and path are
// shared scratch of VR_MAX_WINDOW_ROWS entries, n_s and bad_s shared ints.
// Returns len, or -1 (H empty) when the parent array is not topological.

template <int NT>
__device__ int assemble_history(const ReqDev& rq, int end_node, int32_t* H, int32_t* par,
                                int32_t* path, int* n_s, int* bad_s) {
  const int tid = threadIdx.x, nn = rq.n_nodes;
  for (int j = tid; j < nn; j += NT) par[j] = rq.parent ? rq.parent[j] : j - 1;
  block_sync();
  if (tid == 0) {
    int n = 0, node = end_node, bad = 0;
    while (node >= 0) {
      if (node >= nn) {
        bad = 1;
        break;
      }
      path[n++] = node;
      const int p = par[node];
      if (p >= node || p < -1) {
        bad = 1;
        break;
      }
      node = p;
    }
    *n_s = n;
    *bad_s = bad;
  }
  block_sync();
  const int bad = *bad_s;
  const int from_path = bad ? 0 : min(*n_s, rq.pol.window);
  const int from_hist = bad ? 0 : min(rq.hist_len, rq.pol.window - from_path);
  for (int i = tid; i < from_hist; i += NT) H[i] = rq.hist[rq.hist_len - from_hist + i];
  // path[] is leaf-first
  for (int i = tid; i < from_path; i += NT) H[from_hist + i] = rq.tokens[path[from_path - 1 - i]];
  block_sync();
  return bad ? -1 : from_hist + from_path;
}

// ---------------------------------------------------------------------------
// penalties: one float32 op at a time, round to nearest.

__device__ __forceinline__ float penalize_value(float x, int count, const vr_policy& p) {
  if (p.repeat != 1.f) x = (x > 0.f) ? __fdiv_rn(x, p.repeat) : __fmul_rn(x, p.repeat);
  if (p.frequency != 0.f) x = __fsub_rn(x, __fmul_rn(static_cast<float>(count), p.frequency));
  if (p.presence != 0.f) x = __fsub_rn(x, p.presence);
  return x;
}

// ---------------------------------------------------------------------------
// sampler policy on one pool (values in pool order), run by one warp.
// The e_j are computed by the lanes; one lane then forms the running sums
// pc[j] = e_0 + ... + e_j in pool order, one rounding per addition (the
// sequential sums the policy is defined with).  Every later step reads them:
// top-p's total over the min-p survivors is pc[m-1], its cut is the first j
// with pc[j] >= top_p * pc[m-1], the final S is pc[m-1] of the kept prefix,
// and a draw takes the first j with pc[j] > u * S.  e and pc have room for
// kPool entries; e past the kept count is set to 0.

__device__ __forceinline__ int topk_limit(int32_t top_k) {
  if (top_k < 0) return kTopKAbsent;
  if (top_k == 0) return kPool;
  return top_k < kPool ? top_k : kPool;
}

// smallest j < m with pred(j) over j = lane, lane + 32; -1 if none
template <typename Pred>
__device__ __forceinline__ int warp_first(int m, Pred pred) {
  const int lane = threadIdx.x & 31;
  uint32_t b = __ballot_sync(0xffffffffu, lane < m && pred(lane));
  if (b) return __ffs(b) - 1;
  b = __ballot_sync(0xffffffffu, lane + 32 < m && pred(lane + 32));
  return b ? 32 + __ffs(b) - 1 : -1;
}

// running sums c[j] = w_0 + ... + w_j for j < n <= N, sequential, by one
// lane; w and c are 16-byte aligned arrays of at least N floats.  All N
// weights are read first (no load waits inside the chain of additions);
// entries past n count as zero, so c[j] for n <= j < N repeats c[n - 1];
// c past N is not written.
template <int N>
__device__ __forceinline__ void running_sums_n(const float* w, float* c, int n) {
  // one 16-byte chunk at a time, no array: every value stays in a register
  // (a whole-row array was placed in local memory)
  float acc = 0.0f;
#pragma unroll
  for (int j = 0; j < N; j += 4) {
    const float4 t = *reinterpret_cast<const float4*>(w + j);
    float4 o;
    acc = __fadd_rn(acc, j < n ? t.x : 0.0f);
    o.x = acc;
    acc = __fadd_rn(acc, j + 1 < n ? t.y : 0.0f);
    o.y = acc;
    acc = __fadd_rn(acc, j + 2 < n ? t.z : 0.0f);
    o.z = acc;
    acc = __fadd_rn(acc, j + 3 < n ? t.w : 0.0f);
    o.w = acc;
    *reinterpret_cast<float4*>(c + j) = o;
  }
}

__device__ __forceinline__ void running_sums(const float* w, float* c, int n) {
  // the shortest chain of additions that covers n (c past it is not read)
  if (n <= 8)
    running_sums_n<8>(w, c, n);
  else if (n <= 16)
    running_sums_n<16>(w, c, n);
  else if (n <= 32)
    running_sums_n<32>(w, c, n);
  else
    running_sums_n<64>(w, c, n);
}

// e and pc must be 16-byte aligned shared arrays of kPool floats
// pol by value: its fields live in registers for the whole function
__device__ __forceinline__ void policy_warp(const float* vals, int n, const vr_policy pol,
                                            float* e, float* pc, int* m_out, float* S_out) {
  const int lane = threadIdx.x & 31;
  int K = topk_limit(pol.top_k);
  if (K > n) K = n;
  if (pol.temperature == 0.f) {
    for (int j = lane; j < kPool; j += 32) {
      e[j] = (j == 0) ? 1.0f : 0.0f;
      pc[j] = 1.0f;
    }
    __syncwarp();
    if (lane == 0) {
      *m_out = 1;
      *S_out = 1.0f;
    }
    __syncwarp();
    return;
  }
  const float T = pol.temperature;
  const float v0 = vals[0];
  // entry lane, and entry lane + 32 only when the kept count reaches past
  // 32 (a warp-uniform test); no branches inside an entry
  auto weight = [&](int j) {
    const float v = vals[j];
    const float z = __fdiv_rn(__fsub_rn(v, v0), T);
    const bool live = (j >= 1) & (j < K) & !isnan(v) & (v != -__int_as_float(0x7f800000)) &
                      (z >= -87.0f);
    const float ex = vexp(z);
    return j == 0 ? 1.0f : (live ? ex : 0.0f);
  };
  e[lane] = weight(lane);
  e[lane + 32] = K > 32 ? weight(lane + 32) : 0.0f;
  __syncwarp();
  if (lane == 0) running_sums(e, pc, K);
  __syncwarp();
  int m = K;
  if (pol.min_p > 0.f) {
    const float mp = pol.min_p;
    const int j = warp_first(K, [&](int i) { return i >= 1 && e[i] < mp; });
    if (j >= 1) m = j;
  }
  if (pol.top_p < 1.f) {
    const float thr = __fmul_rn(pol.top_p, pc[m - 1]);
    const int j = warp_first(m, [&](int i) { return pc[i] >= thr; });
    if (j >= 0) m = j + 1;
  }
  __syncwarp();
  for (int j = lane; j < kPool; j += 32)
    if (j >= m) e[j] = 0.0f;
  if (lane == 0) {
    *m_out = m;
    *S_out = pc[m - 1];
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------
// programmatic dependent launch.  Every kernel of the library waits for its
// predecessor grid to complete (wait) before it touches any buffer that a
// predecessor may write or read, and lets the next kernel on the stream
// start launching early (launch_dependents): at once, except the
// projections, which trigger only after their own wait.  So every kernel
// after a window's projection starts after everything before the window is
// complete and may read the window's inputs (drafts, candidates, parents)
// before its own wait, as the row sampling kernel does.  Before their wait
// the projections touch only the weights, which no kernel of a window
// writes; so the kernels that precede them in a window (the host-input
// staging kernel, the split passes) trigger at once.  Completion still follows
// stream order; only launch latency, prologues and the first weight loads
// overlap.  Without the launch attribute both are no-ops.

__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

__host__ __device__ __forceinline__ size_t align_up(size_t x, size_t a) {
  return (x + a - 1) / a * a;
}

}  // namespace vr
