// Candidate pool of every verify row: the top 64 entries in the order
// (value descending, token id ascending), NaN lowest and -0.0 below +0.0
// ("Speculative decoding on RDNA" §03: a 64-wide pool with a fixed tie
// order; "feat(dflash) ...": a top-K select held to byte identity with
// ties, NaN and -inf, re-gridded so that a row is not left to one block).
//
// Each entry becomes one 64-bit composite, (order key << 32) | ~id, so the
// pool order is plain unsigned order of distinct integers and the top 64
// set is unique.  Phase A: grid (segments, rows); a CTA reduces its
// 2048-entry sub-blocks to their top 64 by a block radix select (see
// block_top64).  Phase B:
// one CTA per row merges the segments' candidates the same way, orders the
// 64 survivors by rank counting and gathers the values' own bits from the
// row.  On the sampling path the same CTA then applies the sampler policy
// to its pool and takes every random decision that belongs to its row.
#include <algorithm>

#include "vr_common.cuh"
#include "vr_kernels.h"

namespace vr {
namespace sel {

constexpr int THREADS = 256;
constexpr int SUB = 2048;            // entries per phase-A sub-block
constexpr int A_ITEMS = SUB / THREADS + 1;   // + one carried candidate (threads < 64)
constexpr int MAX_SEG = 80;
constexpr int B_ITEMS = MAX_SEG * kPool / THREADS;   // 20

constexpr int NPASS = 6;
__constant__ int kDigitBits[NPASS] = {12, 12, 8, 12, 12, 8};   // 64 bits, most significant first
constexpr int MAX_BINS = 4096;
constexpr int GATHER_MAX = THREADS;

struct SelectShared {
  uint32_t hist[MAX_BINS];
  uint64_t gather[GATHER_MAX];
  uint64_t out[kPool];
  uint32_t warp_sum[THREADS / 32];
  int count, gcount, digit, above, n_valid;
};

// Block-wide exclusive scan of one value per thread (thread 0 first).
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, SelectShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sh.warp_sum[warp] = incl;
  __syncthreads();
  uint32_t before = 0;
  for (int w = 0; w < warp; ++w) before += sh.warp_sum[w];
  __syncthreads();
  return before + incl - v;
}

// Top-64 of the nonzero composites held by the block (ITEMS per thread).
// Leaves them, in no particular order, in sh.out[0..sh.count).
//
// Radix select on the 64-bit composites, most significant digit first:
// a pass histograms the digit of the entries that still tie with the
// resolved prefix and finds the digit d holding the need-th largest.  The
// first digit is 12 bits wide, so a row's largest values spread over many
// bins.  As soon as the entries tying on d are few (<= 256) they are
// gathered and the remaining choice is made by rank counting; if they are
// exactly the ones still needed, all are taken.
template <int ITEMS>
__device__ void block_top64(const uint64_t (&x)[ITEMS], SelectShared& sh) {
  const int tid = threadIdx.x, lane = tid & 31;
  int mine = 0;
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) mine += (x[i] != 0ull);
  if (tid == 0) {
    sh.n_valid = 0;
    sh.count = 0;
    sh.gcount = 0;
  }
  __syncthreads();
  mine = __reduce_add_sync(0xffffffffu, mine);
  if (lane == 0) atomicAdd(&sh.n_valid, mine);
  __syncthreads();

  uint64_t prefix = 0ull, mask = 0ull;
  bool gathered = false;
  int need = kPool;
  if (sh.n_valid > kPool) {
    int shift = 64;
    for (int pass = 0; pass < NPASS; ++pass) {
      const int bits = kDigitBits[pass];
      const int nb = 1 << bits;
      shift -= bits;
      for (int b = tid; b < nb; b += THREADS) sh.hist[b] = 0u;
      __syncthreads();
#pragma unroll
      for (int i = 0; i < ITEMS; ++i)
        if (x[i] != 0ull && (x[i] & mask) == prefix)
          atomicAdd(&sh.hist[static_cast<uint32_t>(x[i] >> shift) & (nb - 1)], 1u);
      __syncthreads();
      // thread t owns the bins [nb - (t+1) per, nb - t per), walked downwards
      const int per = nb / THREADS;
      const int top = nb - tid * per;
      uint32_t mysum = 0;
      for (int b = top - 1; b >= top - per; --b) mysum += sh.hist[b];
      uint32_t cum = block_exclusive_scan(mysum, sh);
      for (int b = top - 1; b >= top - per; --b) {
        const uint32_t h = sh.hist[b];
        if (cum < static_cast<uint32_t>(need) && cum + h >= static_cast<uint32_t>(need)) {
          sh.digit = b;
          sh.above = static_cast<int>(cum);
        }
        cum += h;
      }
      __syncthreads();
      const int d = sh.digit;
      need -= sh.above;
      prefix |= static_cast<uint64_t>(d) << shift;
      mask |= static_cast<uint64_t>(nb - 1) << shift;
      const int tie = static_cast<int>(sh.hist[d]);
      __syncthreads();
      if (tie == need) break;                 // every tying entry is taken
      if (tie <= GATHER_MAX) {
#pragma unroll
        for (int i = 0; i < ITEMS; ++i)
          if (x[i] != 0ull && (x[i] & mask) == prefix) sh.gather[atomicAdd(&sh.gcount, 1)] = x[i];
        __syncthreads();
        gathered = true;
        break;
      }
    }
  }
  if (!gathered) {
    // all entries at or above the resolved prefix (exactly 64, or all of a
    // block that holds no more than 64)
#pragma unroll
    for (int i = 0; i < ITEMS; ++i)
      if (x[i] != 0ull && (x[i] & mask) >= prefix) sh.out[atomicAdd(&sh.count, 1)] = x[i];
  } else {
#pragma unroll
    for (int i = 0; i < ITEMS; ++i)
      if (x[i] != 0ull && (x[i] & mask) > prefix) sh.out[atomicAdd(&sh.count, 1)] = x[i];
    const int g = sh.gcount;
    if (tid < g) {
      const uint64_t me = sh.gather[tid];
      int rank = 0;
      for (int j = 0; j < g; ++j) rank += (sh.gather[j] > me);
      if (rank < need) sh.out[atomicAdd(&sh.count, 1)] = me;
    }
  }
  __syncthreads();
}

__device__ __forceinline__ uint64_t composite_at(const float* row, long long e, int vocab) {
  if (e >= vocab) return 0ull;
  return pack_key_id(float_key(row[e]), static_cast<uint32_t>(e));
}

__global__ void __launch_bounds__(THREADS)
    select_phase_a(const float* __restrict__ logits, int vocab, int seg_len, int nseg,
                   uint64_t* __restrict__ cand) {
  __shared__ SelectShared sh;
  const int seg = blockIdx.x, row = blockIdx.y, tid = threadIdx.x;
  const float* rp = logits + static_cast<size_t>(row) * vocab;
  const long long s0 = static_cast<long long>(seg) * seg_len;
  const long long s1 = std::min<long long>(s0 + seg_len, vocab);
  uint64_t carry = 0ull;
  for (long long b = s0; b < s1; b += SUB) {
    uint64_t x[A_ITEMS];
#pragma unroll
    for (int i = 0; i < SUB / THREADS; ++i) {
      const long long e = b + i * THREADS + tid;
      x[i] = (e < s1) ? composite_at(rp, e, vocab) : 0ull;
    }
    x[A_ITEMS - 1] = carry;
    block_top64(x, sh);
    carry = (tid < sh.count) ? sh.out[tid] : 0ull;
    __syncthreads();
  }
  if (tid < kPool) cand[(static_cast<size_t>(row) * nseg + seg) * kPool + tid] = carry;
}

// Per-row random decisions of a window, all taken inside the row's own CTA
// so that rows proceed in parallel:
//   argmax: pool[0]
//   y: the row's emit draw from p with u(row, emit)
//   z: the residual draw from (p - q)+ with the same uniform (rows that
//      verify a chain draft with candidates; y if the residual is zero)
//   acc: the accept test u(row, accept) * q(x) < p(x) for the row's draft x
struct RowShared {
  float e[kPool], pc[kPool], r[kPool], pr[kPool];
  float qe[kPool], qp[kQCand];
  float vals[kPool], qv[kQCand];
  int32_t ids[kPool], qid[kQCand];
  int m, qm, chain, acc;
  float S, qS;
};

__device__ __forceinline__ int first_above(const float* c, int m, float t) {
  // smallest j < m with c[j] > t, c non-decreasing; -1 if none
  const int lane = threadIdx.x & 31;
  uint32_t b = __ballot_sync(0xffffffffu, lane < m && c[lane] > t);
  if (b) return __ffs(b) - 1;
  b = __ballot_sync(0xffffffffu, lane + 32 < m && c[lane + 32] > t);
  return b ? 32 + __ffs(b) - 1 : -1;
}

__device__ __forceinline__ int last_positive(const float* w, int m) {
  const int lane = threadIdx.x & 31;
  uint32_t b = __ballot_sync(0xffffffffu, lane + 32 < m && w[lane + 32] > 0.0f);
  if (b) return 32 + 31 - __clz(b);
  b = __ballot_sync(0xffffffffu, lane < m && w[lane] > 0.0f);
  return b ? 31 - __clz(b) : 0;
}

__global__ void __launch_bounds__(THREADS)
    select_phase_b(const float* __restrict__ logits, int vocab, int nseg,
                   const uint64_t* __restrict__ cand, int32_t* __restrict__ pool_ids,
                   float* __restrict__ pool_vals, ReqTable tab, int decide,
                   int4* __restrict__ dec) {
  __shared__ SelectShared sh;
  __shared__ RowShared rs;
  const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint64_t x[B_ITEMS];
  const uint64_t* c = cand + static_cast<size_t>(row) * nseg * kPool;
#pragma unroll
  for (int i = 0; i < B_ITEMS; ++i) {
    const int k = i * THREADS + tid;
    x[i] = (k < nseg * kPool) ? c[k] : 0ull;
  }
  block_top64(x, sh);
  const int n = sh.count;                           // = min(64, vocab)
  if (tid < kPool) {
    int32_t id = -1;
    float v = __int_as_float(0x7fffffff);
    int pos = tid;
    if (tid < n) {
      const uint64_t me = sh.out[tid];
      int rank = 0;
      for (int j = 0; j < n; ++j) rank += (sh.out[j] > me);
      id = static_cast<int32_t>(packed_id(me));
      v = logits[static_cast<size_t>(row) * vocab + id];
      pos = rank;
    }
    pool_ids[static_cast<size_t>(row) * kPool + pos] = id;
    pool_vals[static_cast<size_t>(row) * kPool + pos] = v;
    rs.ids[pos] = id;
    rs.vals[pos] = v;
  }
  if (!decide) return;
  const ReqDev& rq = request(tab, request_of_row(tab, row));
  const vr_policy& pol = rq.pol;
  const int local = row - rq.row0;
  if (pol.temperature == 0.f) {
    __syncthreads();
    if (tid == 0) dec[row] = make_int4(rs.ids[0], rs.ids[0], rs.ids[0], 0);
    return;
  }
  if (tid == 0) rs.chain = 1;
  __syncthreads();
  if (rq.parent)
    for (int j = tid; j < rq.n_nodes; j += THREADS)
      if (rq.parent[j] != j - 1) rs.chain = 0;
  __syncthreads();
  const bool reject_row = rq.q_ids != nullptr && rs.chain && local < rq.n_nodes;
  const uint64_t urow = static_cast<uint64_t>(local);

  if (warp == 0) {
    policy_warp(rs.vals, n, pol, rs.e, &rs.m, &rs.S);
    if (lane == 0) {
      float acc = 0.0f;
      for (int j = 0; j < rs.m; ++j) {
        acc = __fadd_rn(acc, rs.e[j]);
        rs.pc[j] = acc;
      }
    }
  } else if (warp == 1 && reject_row) {
    // q: the node's candidates in pool order, then the same policy
    const float* qv = rq.q_pen + static_cast<size_t>(local) * kQCand;
    const int32_t* qi = rq.q_ids + static_cast<size_t>(local) * kQCand;
    if (lane < kQCand) {
      const uint32_t k = float_key(qv[lane]);
      const int32_t id = qi[lane];
      int rank = 0;
      for (int s2 = 0; s2 < kQCand; ++s2) {
        const uint32_t ks = float_key(qv[s2]);
        const int32_t is = qi[s2];
        rank += (ks > k) || (ks == k && (is < id || (is == id && s2 < lane)));
      }
      rs.qid[rank] = id;
      rs.qv[rank] = qv[lane];
    }
    __syncwarp();
    policy_warp(rs.qv, kQCand, pol, rs.qe, &rs.qm, &rs.qS);
    if (lane < rs.qm) rs.qp[lane] = __fdiv_rn(rs.qe[lane], rs.qS);
  }
  __syncthreads();
  if (warp != 0) return;

  const int m = rs.m;
  const float S = rs.S;
  const float u2 = uniform01(rq.seed, rq.position, urow, kPurposeEmit);
  int j = first_above(rs.pc, m, __fmul_rn(u2, S));
  if (j < 0) j = last_positive(rs.e, m);
  const int32_t y = rs.ids[j];
  int32_t z = y;
  int acc = 0;
  if (reject_row) {
    const int32_t xd = rq.tokens[local];
    const int qm = rs.qm;
    // residual (p - q)+ over the kept entries; p(x) from the matching entry
    float px = 0.0f;
    for (int jj = lane; jj < m; jj += 32) {
      const float pj = __fdiv_rn(rs.e[jj], S);
      float qj = 0.0f;
      for (int s2 = 0; s2 < qm; ++s2)
        if (rs.qid[s2] == rs.ids[jj]) qj = __fadd_rn(qj, rs.qp[s2]);
      const float d = __fsub_rn(pj, qj);
      rs.r[jj] = d > 0.0f ? d : 0.0f;
      if (rs.ids[jj] == xd) px = pj;
    }
    // pool ids are distinct: at most one lane holds p(x)
    for (int o = 16; o >= 1; o >>= 1) {
      const float other = __shfl_xor_sync(0xffffffffu, px, o);
      px = other != 0.0f ? other : px;
    }
    __syncwarp();
    if (lane == 0) {
      float qx = 0.0f;
      for (int s2 = 0; s2 < qm; ++s2)
        if (rs.qid[s2] == xd) qx = __fadd_rn(qx, rs.qp[s2]);
      const float u1 = uniform01(rq.seed, rq.position, urow, kPurposeAccept);
      rs.acc = (qx > 0.0f) ? (__fmul_rn(u1, qx) < px) : (px > 0.0f);
      float a = 0.0f;
      for (int jj = 0; jj < m; ++jj) {
        a = __fadd_rn(a, rs.r[jj]);
        rs.pr[jj] = a;
      }
    }
    __syncwarp();
    acc = rs.acc;
    const float sr = m ? rs.pr[m - 1] : 0.0f;
    if (sr > 0.0f) {
      int jz = first_above(rs.pr, m, __fmul_rn(u2, sr));
      if (jz < 0) jz = last_positive(rs.r, m);
      z = rs.ids[jz];
    }
  }
  if (lane == 0) dec[row] = make_int4(rs.ids[0], y, z, acc);
}

__global__ void policy_kernel(const float* __restrict__ pool_vals, int pool_len, vr_policy pol,
                              int32_t* __restrict__ out_m, float* __restrict__ out_e,
                              float* __restrict__ out_S) {
  __shared__ float vals[kPool];
  __shared__ float e[kPool];
  __shared__ int m;
  __shared__ float S;
  const int row = blockIdx.x;
  for (int j = threadIdx.x; j < kPool; j += 32) vals[j] = pool_vals[static_cast<size_t>(row) * kPool + j];
  __syncwarp();
  policy_warp(vals, pool_len, pol, e, &m, &S);
  for (int j = threadIdx.x; j < kPool; j += 32) out_e[static_cast<size_t>(row) * kPool + j] = e[j];
  if (threadIdx.x == 0) {
    out_m[row] = m;
    out_S[row] = S;
  }
}

}  // namespace sel

int select_segments(int vocab) {
  int nseg = std::min((vocab + sel::SUB - 1) / sel::SUB, sel::MAX_SEG);
  const long long per = (static_cast<long long>(vocab) + nseg - 1) / nseg;
  const long long seg_len = (per + sel::SUB - 1) / sel::SUB * sel::SUB;
  return static_cast<int>((vocab + seg_len - 1) / seg_len);
}

size_t select_cand_bytes(int rows, int vocab) {
  return static_cast<size_t>(rows) * select_segments(vocab) * kPool * sizeof(uint64_t);
}

int launch_select(const float* logits, int rows, int vocab, uint64_t* cand, int32_t* pool_ids,
                  float* pool_vals, const ReqTable* tab, int4* dec, cudaStream_t stream) {
  const int nseg = select_segments(vocab);
  const long long per = (static_cast<long long>(vocab) + nseg - 1) / nseg;
  const int seg_len = static_cast<int>((per + sel::SUB - 1) / sel::SUB * sel::SUB);
  sel::select_phase_a<<<dim3(nseg, rows), sel::THREADS, 0, stream>>>(logits, vocab, seg_len, nseg,
                                                                     cand);
  ReqTable none{};
  sel::select_phase_b<<<rows, sel::THREADS, 0, stream>>>(logits, vocab, nseg, cand, pool_ids,
                                                         pool_vals, tab ? *tab : none,
                                                         tab ? 1 : 0, dec);
  return cudaGetLastError() == cudaSuccess ? VR_OK : VR_ERR_CUDA;
}

int launch_policy(const float* pool_vals, int rows, int pool_len, const vr_policy& pol,
                  int32_t* out_m, float* out_e, float* out_S, cudaStream_t stream) {
  sel::policy_kernel<<<rows, 32, 0, stream>>>(pool_vals, pool_len, pol, out_m, out_e, out_S);
  return cudaGetLastError() == cudaSuccess ? VR_OK : VR_ERR_CUDA;
}

}  // namespace vr
