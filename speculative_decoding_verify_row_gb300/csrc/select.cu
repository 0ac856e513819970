// Candidate pool of every verify row: the top 64 entries in the order
// (value descending, token id ascending), NaN lowest and -0.0 below +0.0
// ("Speculative decoding on RDNA" §03: a 64-wide pool with a fixed tie
// order; "feat(dflash) ...": a top-K select held to byte identity with
// ties, NaN and -inf, re-gridded so that a row is not left to one block).
//
// Each entry becomes one 64-bit composite, (order key << 32) | ~id, so the
// pool order is plain unsigned order of distinct integers and the top 64
// set is unique.  Phase A: grid (segments, rows); a CTA reduces its
// 2048-entry sub-blocks to their top 64 by a block radix select (8-bit
// digits, most significant first, stopping once the candidates that tie on
// the digits resolved so far are exactly the ones still needed).  Phase B:
// one CTA per row merges the segments' candidates the same way, orders the
// 64 survivors by rank counting, gathers the values' own bits from the row,
// and (for the fused path) applies the sampler policy to the pool.
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

struct SelectShared {
  uint32_t hist[256];
  uint64_t out[kPool];
  int count;
  int digit;
  int above;
  int n_valid;
};

// Top-64 of the nonzero composites held by the block (ITEMS per thread).
// Leaves them, in no particular order, in sh.out[0..sh.count).
template <int ITEMS>
__device__ void block_top64(const uint64_t (&x)[ITEMS], SelectShared& sh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int mine = 0;
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) mine += (x[i] != 0ull);
  if (tid == 0) {
    sh.n_valid = 0;
    sh.count = 0;
  }
  __syncthreads();
  mine = __reduce_add_sync(0xffffffffu, mine);
  if (lane == 0) atomicAdd(&sh.n_valid, mine);
  __syncthreads();

  uint64_t prefix = 0ull, mask = 0ull;
  if (sh.n_valid > kPool) {
    int need = kPool;
    for (int pass = 0; pass < 8; ++pass) {
      const int shift = 56 - 8 * pass;
      sh.hist[tid] = 0u;                      // THREADS == 256 bins
      __syncthreads();
#pragma unroll
      for (int i = 0; i < ITEMS; ++i)
        if (x[i] != 0ull && (x[i] & mask) == prefix)
          atomicAdd(&sh.hist[static_cast<uint32_t>(x[i] >> shift) & 255u], 1u);
      __syncthreads();
      if (warp == 0) {
        uint32_t c[8];
        uint32_t tot = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          c[i] = sh.hist[255 - 8 * lane - i];
          tot += c[i];
        }
        uint32_t incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        uint32_t cum = incl - tot;          // entries in higher bins
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (cum < static_cast<uint32_t>(need) && cum + c[i] >= static_cast<uint32_t>(need)) {
            sh.digit = 255 - 8 * lane - i;
            sh.above = static_cast<int>(cum);
          }
          cum += c[i];
        }
      }
      __syncthreads();
      const int d = sh.digit;
      need -= sh.above;
      prefix |= static_cast<uint64_t>(d) << shift;
      mask |= 255ull << shift;
      const bool done = static_cast<int>(sh.hist[d]) == need;
      __syncthreads();
      if (done) break;
    }
  }
#pragma unroll
  for (int i = 0; i < ITEMS; ++i)
    if (x[i] != 0ull && (x[i] & mask) >= prefix) sh.out[atomicAdd(&sh.count, 1)] = x[i];
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

__global__ void __launch_bounds__(THREADS)
    select_phase_b(const float* __restrict__ logits, int vocab, int nseg,
                   const uint64_t* __restrict__ cand, int32_t* __restrict__ pool_ids,
                   float* __restrict__ pool_vals, ReqTable tab, int with_policy,
                   double* __restrict__ pol_e, int32_t* __restrict__ pol_m,
                   double* __restrict__ pol_S) {
  __shared__ SelectShared sh;
  __shared__ float vals[kPool];
  const int row = blockIdx.x, tid = threadIdx.x;
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
    if (tid < n) {
      const uint64_t me = sh.out[tid];
      int rank = 0;
      for (int j = 0; j < n; ++j) rank += (sh.out[j] > me);
      id = static_cast<int32_t>(packed_id(me));
      v = logits[static_cast<size_t>(row) * vocab + id];
      pool_ids[static_cast<size_t>(row) * kPool + rank] = id;
      pool_vals[static_cast<size_t>(row) * kPool + rank] = v;
      vals[rank] = v;
    } else {
      pool_ids[static_cast<size_t>(row) * kPool + tid] = id;
      pool_vals[static_cast<size_t>(row) * kPool + tid] = v;
      vals[tid] = v;
    }
  }
  if (!with_policy) return;
  __syncthreads();
  if (tid < 32) {
    const ReqDev& rq = request(tab, request_of_row(tab, row));
    __shared__ double e[kPool];
    __shared__ int m;
    __shared__ double S;
    policy_warp(vals, n, rq.pol, e, &m, &S);
    for (int j = tid; j < kPool; j += 32) pol_e[static_cast<size_t>(row) * kPool + j] = e[j];
    if (tid == 0) {
      pol_m[row] = m;
      pol_S[row] = S;
    }
  }
}

__global__ void policy_kernel(const float* __restrict__ pool_vals, int pool_len, vr_policy pol,
                              int32_t* __restrict__ out_m, double* __restrict__ out_e,
                              double* __restrict__ out_S) {
  __shared__ float vals[kPool];
  __shared__ double e[kPool];
  __shared__ int m;
  __shared__ double S;
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
                  float* pool_vals, const ReqTable* tab, double* pol_e, int32_t* pol_m,
                  double* pol_S, cudaStream_t stream) {
  const int nseg = select_segments(vocab);
  const long long per = (static_cast<long long>(vocab) + nseg - 1) / nseg;
  const int seg_len = static_cast<int>((per + sel::SUB - 1) / sel::SUB * sel::SUB);
  sel::select_phase_a<<<dim3(nseg, rows), sel::THREADS, 0, stream>>>(logits, vocab, seg_len, nseg,
                                                                     cand);
  ReqTable none{};
  sel::select_phase_b<<<rows, sel::THREADS, 0, stream>>>(logits, vocab, nseg, cand, pool_ids,
                                                         pool_vals, tab ? *tab : none,
                                                         tab ? 1 : 0, pol_e, pol_m, pol_S);
  return cudaGetLastError() == cudaSuccess ? VR_OK : VR_ERR_CUDA;
}

int launch_policy(const float* pool_vals, int rows, int pool_len, const vr_policy& pol,
                  int32_t* out_m, double* out_e, double* out_S, cudaStream_t stream) {
  sel::policy_kernel<<<rows, 32, 0, stream>>>(pool_vals, pool_len, pol, out_m, out_e, out_S);
  return cudaGetLastError() == cudaSuccess ? VR_OK : VR_ERR_CUDA;
}

}  // namespace vr
