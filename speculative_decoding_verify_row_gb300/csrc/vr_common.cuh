// Device-side building blocks shared by the verifyrow kernels.
//
// Every floating-point step that decides an integer (a pool order, a kept
// count, a draw) uses explicit round-to-nearest intrinsics, so that no
// fused multiply-add or fast-math rewrite can change a bit; the library is
// also compiled with --fmad=false.
#pragma once

#include <cstdint>
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
// key (seed, 0); u = (word0 >> 11) * 2^-53.

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

__device__ __forceinline__ double uniform01(uint64_t seed, uint64_t position, uint64_t row,
                                            uint64_t purpose) {
  const uint64_t w = philox_word0(position, row, purpose, 0ull, seed, 0ull);
  return __dmul_rn(__ull2double_rn(w >> 11), 0x1p-53);
}

// ---------------------------------------------------------------------------
// vexp: Cody-Waite reduction by ln 2 (C1 = ln 2 with its low 32 significand
// bits cleared, C2 = nearest double to ln 2 - C1), degree-13 Taylor
// polynomial of e^r in Horner form (coefficients 1/j! rounded to nearest),
// scaling by 2^n from the exponent bits.  IEEE double +, -, x only.

__device__ __forceinline__ double vexp(double z) {
  if (!(z >= -708.0)) return 0.0;
  if (z > 709.0) return __longlong_as_double(0x7FF0000000000000ll);
  constexpr double kInvLn2 = 0x1.71547652b82fep+0;
  constexpr double kC1 = 0x1.62e4200000000p-1;
  constexpr double kC2 = 0x1.fdf473de6af28p-22;
  const double nf = rint(__dmul_rn(z, kInvLn2));
  const double r = __dsub_rn(__dsub_rn(z, __dmul_rn(nf, kC1)), __dmul_rn(nf, kC2));
  double p = 0x1.6124613a86d09p-33;                    // 1/13!
  p = __dadd_rn(__dmul_rn(p, r), 0x1.1eed8eff8d898p-29);  // 1/12!
  p = __dadd_rn(__dmul_rn(p, r), 0x1.ae64567f544e4p-26);  // 1/11!
  p = __dadd_rn(__dmul_rn(p, r), 0x1.27e4fb7789f5cp-22);  // 1/10!
  p = __dadd_rn(__dmul_rn(p, r), 0x1.71de3a556c734p-19);  // 1/9!
  p = __dadd_rn(__dmul_rn(p, r), 0x1.a01a01a01a01ap-16);  // 1/8!
  p = __dadd_rn(__dmul_rn(p, r), 0x1.a01a01a01a01ap-13);  // 1/7!
  p = __dadd_rn(__dmul_rn(p, r), 0x1.6c16c16c16c17p-10);  // 1/6!
  p = __dadd_rn(__dmul_rn(p, r), 0x1.1111111111111p-7);   // 1/5!
  p = __dadd_rn(__dmul_rn(p, r), 0x1.5555555555555p-5);   // 1/4!
  p = __dadd_rn(__dmul_rn(p, r), 0x1.5555555555555p-3);   // 1/3!
  p = __dadd_rn(__dmul_rn(p, r), 0x1.0000000000000p-1);   // 1/2!
  p = __dadd_rn(__dmul_rn(p, r), 1.0);                    // 1/1!
  p = __dadd_rn(__dmul_rn(p, r), 1.0);                    // 1/0!
  const long long n = static_cast<long long>(nf);
  return __dmul_rn(p, __longlong_as_double((n + 1023ll) << 52));
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
// sampler policy on one pool (values in pool order).  The e_j are computed
// by the calling warp's lanes; lane 0 then runs the sequential min-p, top-p
// and sum, in pool order.  e has room for kPool entries; entries past the
// kept count are set to 0.

__device__ __forceinline__ int topk_limit(int32_t top_k) {
  if (top_k < 0) return kTopKAbsent;
  if (top_k == 0) return kPool;
  return top_k < kPool ? top_k : kPool;
}

__device__ __forceinline__ void policy_warp(const float* vals, int n, const vr_policy& pol,
                                            double* e, int* m_out, double* S_out) {
  const int lane = threadIdx.x & 31;
  int K = topk_limit(pol.top_k);
  if (K > n) K = n;
  if (pol.temperature == 0.f) {
    for (int j = lane; j < kPool; j += 32) e[j] = (j == 0) ? 1.0 : 0.0;
    __syncwarp();
    if (lane == 0) {
      *m_out = 1;
      *S_out = 1.0;
    }
    __syncwarp();
    return;
  }
  const double T = static_cast<double>(pol.temperature);
  const double v0 = static_cast<double>(vals[0]);
  for (int j = lane; j < kPool; j += 32) {
    double ej = 0.0;
    if (j == 0) {
      ej = 1.0;
    } else if (j < K) {
      const float v = vals[j];
      if (!(isnan(v) || v == -__int_as_float(0x7f800000))) {
        const double z = __ddiv_rn(__dsub_rn(static_cast<double>(v), v0), T);
        ej = (z >= -708.0) ? vexp(z) : 0.0;
      }
    }
    e[j] = ej;
  }
  __syncwarp();
  if (lane == 0) {
    int m = K;
    if (pol.min_p > 0.f) {
      const double mp = static_cast<double>(pol.min_p);
      int j = 1;
      while (j < m && e[j] >= mp) ++j;
      m = j;
    }
    if (pol.top_p < 1.f) {
      double s = 0.0;
      for (int j = 0; j < m; ++j) s = __dadd_rn(s, e[j]);
      const double thr = __dmul_rn(static_cast<double>(pol.top_p), s);
      double c = 0.0;
      for (int j = 0; j < m; ++j) {
        c = __dadd_rn(c, e[j]);
        if (c >= thr) {
          m = j + 1;
          break;
        }
      }
    }
    double S = 0.0;
    for (int j = 0; j < m; ++j) S = __dadd_rn(S, e[j]);
    for (int j = m; j < kPool; ++j) e[j] = 0.0;
    *m_out = m;
    *S_out = S;
  }
  __syncwarp();
}

// t = u * S; the first j whose running sum exceeds t; if rounding leaves
// none, the last j with a positive weight.
__device__ __forceinline__ int draw_index(const double* w, int n, double total, double u) {
  const double t = __dmul_rn(u, total);
  double c = 0.0;
  for (int j = 0; j < n; ++j) {
    c = __dadd_rn(c, w[j]);
    if (c > t) return j;
  }
  for (int j = n - 1; j >= 0; --j)
    if (w[j] > 0.0) return j;
  return 0;
}

// p(x) = sum over kept entries holding x of e_j / S, in pool order.
__device__ __forceinline__ double prob_of(const int32_t* ids, const double* e, int m, double S,
                                          int32_t x) {
  double acc = 0.0;
  for (int j = 0; j < m; ++j)
    if (ids[j] == x) acc = __dadd_rn(acc, __ddiv_rn(e[j], S));
  return acc;
}

__host__ __device__ __forceinline__ size_t align_up(size_t x, size_t a) {
  return (x + a - 1) / a * a;
}

}  // namespace vr
