// The sampling stage of a verify window, in one kernel: candidate pools,
// sampler policy, per-row random decisions and acceptance.
//
// Pool ("Speculative decoding on RDNA" §03: a 64-wide pool with a fixed tie
// order; "feat(dflash) ...": a top-K select held to byte identity with ties,
// NaN and -inf).  Each entry of a row becomes one 64-bit composite,
// (order key << 32) | ~id, whose unsigned order is the pool order (value
// descending, token id ascending, NaN lowest, -0.0 below +0.0), so the top-64
// set is unique.
//
// Grid (segments, rows), no CTA ever waits for another:
//  1. every CTA reduces its segment of one row to the segment's top 64 (a
//     threshold filter from per-thread maxima plus rank counting; a block
//     radix select when ties defeat the filter) and stores them in pool
//     order;
//  2. it takes a ticket on the row's counter; the CTA that draws the last
//     ticket has every segment list of the row available, merges them
//     pairwise (merge path) into the row's pool, applies the sampler policy
//     and takes every random decision of the row (emit draw, accept test,
//     residual draw), and resets the counter;
//  3. that CTA then takes a ticket on the request's counter; the last row of
//     the request to finish walks the request's rows and writes the emitted
//     ids (greedy prefix or longest tree branch, §02; rejection sampling,
//     §03 steps 1-4, against the draft candidates' q or, for drafts proposed
//     without probabilities, q = delta(draft), §06; naive descent for
//     deterministic tree drafts, "feat(dflash) ...").
// Tickets follow a __threadfence() after the CTA's writes, so the last CTA
// sees all of them (the usual threadfence-reduction pattern).
#include <algorithm>

#include "vr_common.cuh"
#include "vr_kernels.h"

namespace vr {
namespace smp {

constexpr int THREADS = 256;
constexpr int SUB = 4096;                    // entries per sub-block of a segment
constexpr int ITEMS = SUB / THREADS + 1;     // + one carried candidate (threads < 64)
constexpr int MAX_SEG = 64;
constexpr int NPASS = 6;
__constant__ int kDigitBits[NPASS] = {12, 12, 8, 12, 12, 8};   // 64 bits, most significant first
constexpr int MAX_BINS = 4096;
constexpr int GATHER_MAX = THREADS;
constexpr int MAXR = VR_MAX_WINDOW_ROWS;

struct SelectShared {
  uint32_t hist[MAX_BINS];
  __align__(16) uint64_t gather[GATHER_MAX];
  uint64_t out[kPool];
  uint64_t sorted[kPool];
  uint64_t warp_thr[THREADS / 32];
  uint32_t warp_sum[THREADS / 32];
  int count, gcount, digit, above, n_valid;
};

struct MergeShared {
  uint64_t in[MAX_SEG][kPool];
  uint64_t out[MAX_SEG / 2][kPool];
};

constexpr int PT = 64;                       // entries per thread, one-pass segment select
constexpr int SEG_FAST = THREADS * PT;       // 16384 entries per segment
constexpr int FAST_CAP = 256;                // entries at or above the threshold, at most

struct FastShared {
  uint32_t buf[2][THREADS];
  __align__(16) uint64_t gather[FAST_CAP];
  uint64_t sorted[kPool];
  uint32_t warp_cnt[THREADS / 32];
  uint32_t warp_thr[THREADS / 32];
  uint32_t thr;
};

union StageShared {
  SelectShared sel;
  MergeShared mrg;
  FastShared fast;
};

constexpr int GI_MAX = 20;          // group maxima per thread: vocab <= 32 * 256 * 20
constexpr int C_MAX = kPool * 32;   // candidates of the chosen groups, at most

struct RowsShared {
  union {
    SelectShared sel;
    FastShared fast;
  };
  __align__(16) uint64_t cands[C_MAX];
  uint64_t pool[kPool];
  int ccount;

  // the row's penalty history and what it implies, built before the wait:
  // its distinct in-vocabulary tokens with their counts, and the distinct
  // 32-row groups they fall in
  int32_t H[VR_MAX_PENALTY_WINDOW];
  int32_t par[VR_MAX_WINDOW_ROWS];
  int32_t path[VR_MAX_WINDOW_ROWS];
  int h_len, h_bad;
  int32_t tok_u[VR_MAX_PENALTY_WINDOW];
  int32_t cnt_u[VR_MAX_PENALTY_WINDOW];
  int32_t grp_u[VR_MAX_PENALTY_WINDOW];
  int n_u, n_grp;
};

struct RowShared {
  __align__(16) float e[kPool];
  __align__(16) float pc[kPool];
  __align__(16) float r[kPool];
  __align__(16) float pr[kPool];
  __align__(16) float qe[kPool];
  __align__(16) float qpc[kPool];
  float qp[kQCand];
  float vals[kPool], qv[kQCand];
  int32_t ids[kPool], qid[kQCand];
  int m, qm, chain, acc;
  int32_t draft;
  float S, qS, u1, u2;
  ReqDev req;     // the row's request (load_request), read from here
  int req_b;      // its index in the request table
  int4 dec;       // the row's decisions, as written to dec[row]
  uint32_t acc_bits;   // chains: the accept bits of every row of the request
};

struct AcceptShared {
  int32_t tok[MAXR], par[MAXR];
  int4 d[MAXR];
  int32_t depth[MAXR];       // greedy tree walk: each node's depth and
  uint8_t ok[MAXR];          // whether its whole path agrees
  int bad, not_chain;
};

// ---------------------------------------------------------------------------
// block radix select

// Find the bin holding the need-th largest entry, bins walked from the top.
// Warp w owns the bins [nb - (w+1) nb/8, nb - w nb/8); its lanes read them
// in 32-bin chunks with consecutive lanes on consecutive bins (no bank
// conflicts), a warp scan turns each chunk into running counts, and the
// warps' totals give each warp the count of everything above its range.
__device__ __forceinline__ void find_digit(int nb, int need, SelectShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int per_warp = nb / (THREADS / 32);
  const int top = nb - warp * per_warp;
  uint32_t total = 0;
  for (int c = 0; c < per_warp; c += 32) total += sh.hist[top - 1 - c - lane];
  total = __reduce_add_sync(0xffffffffu, total);
  if (lane == 0) sh.warp_sum[warp] = total;
  block_sync();
  uint32_t cum = 0;
  for (int w = 0; w < warp; ++w) cum += sh.warp_sum[w];
  if (cum < static_cast<uint32_t>(need) && cum + total >= static_cast<uint32_t>(need)) {
    for (int c = 0; c < per_warp; c += 32) {
      const int b = top - 1 - c - lane;          // lane 0 holds the highest bin
      const uint32_t h = sh.hist[b];
      uint32_t incl = h;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const uint32_t before = cum + incl - h;
      if (before < static_cast<uint32_t>(need) && before + h >= static_cast<uint32_t>(need)) {
        sh.digit = b;
        sh.above = static_cast<int>(before);
      }
      cum += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  block_sync();
}

// Top-64 of the nonzero composites held by the block (ITEMS per thread),
// left in no particular order in sh.out[0..sh.count).  Radix select, most
// significant digit first (12-bit first digit, so a row's largest values
// spread over many bins); once the entries that tie with the resolved prefix
// are few (<= 256) they are gathered and the rest is decided by rank
// counting; if they are exactly the ones still needed, all are taken.
template <int N>
__device__ void block_top64(const uint64_t (&x)[N], SelectShared& sh) {
  const int tid = threadIdx.x, lane = tid & 31;
  int mine = 0;
#pragma unroll
  for (int i = 0; i < N; ++i) mine += (x[i] != 0ull);
  if (tid == 0) {
    sh.n_valid = 0;
    sh.count = 0;
    sh.gcount = 0;
  }
  block_sync();
  mine = __reduce_add_sync(0xffffffffu, mine);
  if (lane == 0) atomicAdd(&sh.n_valid, mine);
  block_sync();

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
      block_sync();
#pragma unroll
      for (int i = 0; i < N; ++i)
        if (x[i] != 0ull && (x[i] & mask) == prefix)
          atomicAdd(&sh.hist[static_cast<uint32_t>(x[i] >> shift) & (nb - 1)], 1u);
      block_sync();
      find_digit(nb, need, sh);
      const int d = sh.digit;
      need -= sh.above;
      prefix |= static_cast<uint64_t>(d) << shift;
      mask |= static_cast<uint64_t>(nb - 1) << shift;
      const int tie = static_cast<int>(sh.hist[d]);
      block_sync();
      if (tie == need) break;                 // every tying entry is taken
      if (tie <= GATHER_MAX) {
#pragma unroll
        for (int i = 0; i < N; ++i)
          if (x[i] != 0ull && (x[i] & mask) == prefix) sh.gather[atomicAdd(&sh.gcount, 1)] = x[i];
        block_sync();
        gathered = true;
        break;
      }
    }
  }
  if (!gathered) {
#pragma unroll
    for (int i = 0; i < N; ++i)
      if (x[i] != 0ull && (x[i] & mask) >= prefix) sh.out[atomicAdd(&sh.count, 1)] = x[i];
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i)
      if (x[i] != 0ull && (x[i] & mask) > prefix) sh.out[atomicAdd(&sh.count, 1)] = x[i];
    const int g = sh.gcount;
    if (tid < g) {
      const uint64_t me = sh.gather[tid];
      int rank = 0;
      for (int j = 0; j < g; ++j) rank += (sh.gather[j] > me);
      if (rank < need) sh.out[atomicAdd(&sh.count, 1)] = me;
    }
  }
  block_sync();
}

// cand[0..n) (distinct composites, n <= THREADS; cand 16-byte aligned) ->
// sorted[rank] for the ranks below 64 (sorted zeroed by the caller).  Each
// candidate's rank is counted by q = 4, 2 or 1 threads (as n allows), each
// over every q-th pair of entries, and summed by shuffles.  Pairs are read as
// one 16-byte load, four pairs at a time: each comparison waits on no other.
__device__ __forceinline__ void rank_into(const uint64_t* cand, int n, uint64_t* sorted) {
  const int tid = threadIdx.x;
  const int q = n <= THREADS / 4 ? 4 : (n <= THREADS / 2 ? 2 : 1);
  const int c = tid / q, part = tid % q;
  const uint64_t me = c < n ? cand[c] : 0ull;
  int rank = 0;
  if (c < n) {
    const ulonglong2* pairs = reinterpret_cast<const ulonglong2*>(cand);
    const int np = n >> 1;          // whole pairs; an odd n leaves cand[n - 1]
    int k = part;
    for (; k + 3 * q < np; k += 4 * q) {
      const ulonglong2 p0 = pairs[k], p1 = pairs[k + q], p2 = pairs[k + 2 * q],
                       p3 = pairs[k + 3 * q];
      rank += (p0.x > me) + (p0.y > me) + (p1.x > me) + (p1.y > me) + (p2.x > me) +
              (p2.y > me) + (p3.x > me) + (p3.y > me);
    }
    for (; k < np; k += q) {
      const ulonglong2 p0 = pairs[k];
      rank += (p0.x > me) + (p0.y > me);
    }
    if ((n & 1) && part == np % q) rank += cand[n - 1] > me ? 1 : 0;
  }
  if (q >= 2) rank += __shfl_xor_sync(0xffffffffu, rank, 1);
  if (q >= 4) rank += __shfl_xor_sync(0xffffffffu, rank, 2);
  if (c < n && part == 0 && rank < kPool) sorted[rank] = me;
}

// Descending bitonic sort of one value per lane across a warp.
template <class U>
__device__ __forceinline__ U warp_sort_desc(U v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1)
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const U o = __shfl_xor_sync(0xffffffffu, v, j);
      const bool keep_max = ((lane & k) == 0) == ((lane & j) == 0);
      v = keep_max ? (v > o ? v : o) : (v < o ? v : o);
    }
  return v;
}

// Top-64 of the block's nonzero composites, in pool order, into sh.sorted
// (zero-padded).  Filter first: with t_w the 8th largest of the 32 per-thread
// maxima of warp w, at least 8 entries of every warp reach min_w t_w, so at
// least 64 entries of the block do (or all of them, if fewer exist).  The
// entries at or above that threshold are compacted and ranked against each
// other; rank < 64 is the pool position.  Returns false (nothing written)
// when more than 256 entries pass, e.g. for rows full of ties; the caller
// then falls back to the radix select.
template <int N>
__device__ bool block_top64_filtered(const uint64_t (&x)[N], SelectShared& sh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint64_t mx = 0ull;
#pragma unroll
  for (int i = 0; i < N; ++i) mx = x[i] > mx ? x[i] : mx;
  const uint64_t sorted = warp_sort_desc(mx);
  if (lane == 7) sh.warp_thr[warp] = sorted;
  if (tid == 0) sh.gcount = 0;
  block_sync();
  uint64_t thr = sh.warp_thr[0];
#pragma unroll
  for (int w = 1; w < THREADS / 32; ++w) thr = sh.warp_thr[w] < thr ? sh.warp_thr[w] : thr;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const bool pass = (x[i] != 0ull) & (x[i] >= thr);
    const uint32_t ball = __ballot_sync(0xffffffffu, pass);
    if (ball) {
      int base = 0;
      if (lane == 0) base = atomicAdd(&sh.gcount, __popc(ball));
      base = __shfl_sync(0xffffffffu, base, 0);
      const int pos = base + __popc(ball & ((1u << lane) - 1u));
      if (pass && pos < GATHER_MAX) sh.gather[pos] = x[i];
    }
  }
  block_sync();
  const int n = sh.gcount;
  if (n > GATHER_MAX) return false;
  if (tid < kPool) sh.sorted[tid] = 0ull;
  block_sync();
  rank_into(sh.gather, n, sh.sorted);
  block_sync();
  return true;
}

// The float whose order key is k (the inverse of float_key); NaN, whose key
// is 0 whatever its bits, is read back from the row, so id must be a real
// entry's (never a padding entry's).
__device__ __forceinline__ float value_of_key(uint32_t k, const float* row, int32_t id) {
  if (k == 0u) return __ldcg(row + id);
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

__device__ __forceinline__ uint64_t composite_at(const float* row, long long e) {
  return pack_key_id(float_key(row[e]), static_cast<uint32_t>(e));
}

// Descending bitonic sort of one key per thread across the block: thread t
// ends with the t-th largest.  Partners within a warp exchange by shuffle;
// across warps through shared memory, two buffers used in turn so that one
// barrier per such step suffices.
__device__ __forceinline__ uint32_t block_sort_desc(uint32_t v, uint32_t (&buf)[2][THREADS]) {
  const int tid = threadIdx.x;
  int flip = 0;
#pragma unroll
  for (int k = 2; k <= THREADS; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      uint32_t o;
      if (j >= 32) {
        buf[flip][tid] = v;
        block_sync();
        o = buf[flip][tid ^ j];
        flip ^= 1;
      } else {
        o = __shfl_xor_sync(0xffffffffu, v, j);
      }
      const bool keep_max = ((tid & k) == 0) == ((tid & j) == 0);
      v = keep_max ? max(v, o) : min(v, o);
    }
  }
  return v;
}

// Top 64 of the (key, id) composites the block holds, NI keys per thread,
// into fs.sorted in pool order (zero-padded).  Entry i of thread t is held
// iff i * THREADS < len (len = entries - t) and has id id0 + i * THREADS.
// T = the 64th largest of the 256 per-thread largest keys: 64 threads hold a
// key >= T, so at least 64 entries do, and the top 64 all have keys >= T.
// With kmin < 64 only the first kmin entries of fs.sorted need to be exact:
// T is then the smallest over the warps of each warp's ceil(kmin / 8)-th
// largest per-thread key (one warp sort and one barrier instead of the block
// sort), which at least kmin threads reach.
// The entries with key >= T (usually about 70) are compacted by a block scan
// and ranked as composites.  Returns false (after a barrier, nothing
// written) when more than FAST_CAP entries reach T (many ties at T, or one
// thread holding most of the top); the caller then takes the radix path.
template <int NI>
__device__ bool keys_top64(const uint32_t (&key)[NI], int len, uint32_t id0, FastShared& fs,
                           int kmin = kPool) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the thread's largest held key, by a reduction tree (unheld keys are 0)
  uint32_t m[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) m[i] = i * THREADS < len ? key[i] : 0u;
#pragma unroll
  for (int w = 1; w < NI; w <<= 1)
#pragma unroll
    for (int i = 0; i + w < NI; i += 2 * w) m[i] = max(m[i], m[i + w]);
  uint32_t thr;
  if (kmin >= kPool) {
    const uint32_t T = block_sort_desc(m[0], fs.buf);
    if (tid == kPool - 1) fs.thr = T;
    block_sync();
    thr = fs.thr;
  } else {
    const uint32_t srt = warp_sort_desc(m[0]);
    if (lane == (kmin + 7) / 8 - 1) fs.warp_thr[warp] = srt;
    block_sync();
    thr = fs.warp_thr[0];
#pragma unroll
    for (int w = 1; w < THREADS / 32; ++w) thr = fs.warp_thr[w] < thr ? fs.warp_thr[w] : thr;
  }
  // held entries with key >= thr (bitwise tests: no branches)
  uint32_t cnt = 0;
#pragma unroll
  for (int i = 0; i < NI; ++i) cnt += ((i * THREADS < len) & (key[i] >= thr)) ? 1u : 0u;
  uint32_t incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) fs.warp_cnt[warp] = incl;
  block_sync();
  uint32_t off = incl - cnt, total = 0;
#pragma unroll
  for (int w = 0; w < THREADS / 32; ++w) {
    const uint32_t t = fs.warp_cnt[w];
    off += (w < warp) ? t : 0u;
    total += t;
  }
  if (total > static_cast<uint32_t>(FAST_CAP)) {
    block_sync();
    return false;
  }
  if (cnt) {
#pragma unroll
    for (int i = 0; i < NI; ++i)
      if ((i * THREADS < len) & (key[i] >= thr))
        fs.gather[off++] = pack_key_id(key[i], id0 + static_cast<uint32_t>(i * THREADS));
  }
  if (tid < kPool) fs.sorted[tid] = 0ull;
  block_sync();
  rank_into(fs.gather, static_cast<int>(total), fs.sorted);
  block_sync();
  return true;
}

// Top 64 of one segment [s0, s1) of at most SEG_FAST entries in one pass
// (keys_top64 on the row's float keys; thread t holds s0 + i * THREADS + t).
__device__ bool segment_top64_fast(const float* __restrict__ rp, long long s0, long long s1,
                                   FastShared& fs, int kmin = kPool) {
  const int tid = threadIdx.x;
  const int n_seg = static_cast<int>(s1 - s0);
  // every load is unconditional (entries past the segment read its first
  // entry and are masked), so all PT loads are in flight together
  float v[PT];
#pragma unroll
  for (int i = 0; i < PT; ++i) {
    const int e = i * THREADS + tid;
    v[i] = ld_logit(rp + s0 + (e < n_seg ? e : 0));
  }
  uint32_t key[PT];
#pragma unroll
  for (int i = 0; i < PT; ++i) key[i] = float_key(v[i]);
  return keys_top64(key, n_seg - tid, static_cast<uint32_t>(s0) + static_cast<uint32_t>(tid), fs,
                    kmin);
}

// ---------------------------------------------------------------------------
// merge of sorted lists

// The (k+1)-th largest of two descending lists of 64 distinct nonzero
// composites padded with zeros: merge path, i.e. the number i of entries
// that come from a among the first k outputs, found by binary search.
__device__ __forceinline__ uint64_t merged_at(const uint64_t* a, const uint64_t* b, int k) {
  int lo = k > kPool ? k - kPool : 0, hi = k < kPool ? k : kPool;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (a[mid] > b[k - 1 - mid]) lo = mid + 1;
    else hi = mid;
  }
  const int i = lo;
  return (i < kPool && (k - i >= kPool || a[i] > b[k - i])) ? a[i] : b[k - i];
}

// Merge the row's nseg sorted lists (each the top 64 of its segment) into
// the row's top 64, in pool order.  Returns the list (shared memory).
// Pairwise merge path: the top 64 of the union of two lists is the top 64 of
// their merge, and each output position is found by a binary search, so
// ceil(log2(nseg)) rounds of independent searches give the pool.
__device__ const uint64_t* merge_lists(const uint64_t* lists, int nseg, MergeShared& ms) {
  const int tid = threadIdx.x;
  const int total = nseg * kPool;
  for (int base = 0; base < total; base += 4 * THREADS) {
    uint64_t t[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = base + u * THREADS + tid;
      t[u] = __ldcg(lists + (i < total ? i : 0));    // unconditional: loads overlap
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = base + u * THREADS + tid;
      if (i < total) ms.in[i / kPool][i % kPool] = t[u];
    }
  }
  block_sync();
  uint64_t(*src)[kPool] = ms.in;
  uint64_t(*dst)[kPool] = ms.out;
  int nl = nseg;
  while (nl > 1) {
    const int pairs = nl >> 1;
    for (int i = tid; i < pairs * kPool; i += THREADS) {
      const int p = i / kPool, k = i % kPool;
      dst[p][k] = merged_at(src[2 * p], src[2 * p + 1], k);
    }
    if (nl & 1)
      for (int k = tid; k < kPool; k += THREADS) dst[pairs][k] = src[nl - 1][k];
    block_sync();
    uint64_t(*t)[kPool] = src;
    src = dst;
    dst = t;
    nl = pairs + (nl & 1);
  }
  return src[0];
}

// The row's top k (k <= RM_K, nseg <= RM_SEG) from the first k entries of
// each segment's list: an entry at position j of list a ranks j plus, for
// every other list, the number of its first k entries above it (each list
// descends, zeros last, so that number is found by a fixed five-step binary
// search; the searches of all lists run side by side).  Composites are
// distinct, so the ranks are; entries of rank < k land in out[rank].  One
// barrier instead of a merge round per halving.  Returns the pool (k
// entries, zero-padded to 64).
constexpr int RM_K = 16, RM_SEG = 16;
__device__ const uint64_t* rank_merge(const uint64_t* lists, int nseg, int k, MergeShared& ms) {
  const int tid = threadIdx.x;
  const int a = tid / RM_K, j = tid % RM_K;                // nseg * RM_K <= THREADS
  const bool mine = a < nseg && j < k;
  uint64_t c = 0ull;
  if (mine) c = __ldcg(lists + static_cast<size_t>(a) * kPool + j);
  if (a < RM_SEG) ms.in[a][j] = mine ? c : 0ull;           // slots past k read as zero
  if (tid < kPool) ms.out[0][tid] = 0ull;
  block_sync();
  if (mine && c != 0ull) {
    int rank = j;
#pragma unroll
    for (int b = 0; b < RM_SEG; ++b) {
      int lo = 0;
#pragma unroll
      for (int step = RM_K; step > 0; step >>= 1)
        if (lo + step <= k && ms.in[b][lo + step - 1] > c) lo += step;
      rank += (b < nseg && b != a) ? lo : 0;
    }
    if (rank < k) ms.out[0][rank] = c;
  }
  block_sync();
  return ms.out[0];
}

// ---------------------------------------------------------------------------
// per-row decisions

// Copy the request of `row`, and its index, into rs.req / rs.req_b: one
// round of loads by the first warp.  Every later read of a request field is
// then a shared-memory read, not a dependent load from the kernel's
// parameter buffer or the workspace (each of those cost a memory latency
// when first touched after the wait).  Ends with a block barrier.
__device__ __forceinline__ void load_request(const ReqTable& tab, int row, RowShared& rs) {
  constexpr int W = static_cast<int>(sizeof(ReqDev) / 4);
  static_assert(sizeof(ReqDev) % 4 == 0 && W <= 64, "request copy");
  const int tid = threadIdx.x;
  if (tid < 32) {
    const int b = request_of_row(tab, row);
    const uint32_t* src = reinterpret_cast<const uint32_t*>(&request(tab, b));
    uint32_t* dst = reinterpret_cast<uint32_t*>(&rs.req);
    const uint32_t w0 = src[tid];
    const uint32_t w1 = tid + 32 < W ? src[tid + 32] : 0u;
    if (tid < W) dst[tid] = w0;
    if (tid + 32 < W) dst[tid + 32] = w1;
    if (tid == 0) rs.req_b = b;
  }
  block_sync();
}

__device__ __forceinline__ int last_positive(const float* w, int m) {
  const int lane = threadIdx.x & 31;
  uint32_t b = __ballot_sync(0xffffffffu, lane + 32 < m && w[lane + 32] > 0.0f);
  if (b) return 32 + 31 - __clz(b);
  b = __ballot_sync(0xffffffffu, lane < m && w[lane] > 0.0f);
  return b ? 31 - __clz(b) : 0;
}

// All random decisions of one row, taken from its pool (rs.ids/rs.vals, n
// entries) by the whole CTA; writes dec[row] = (argmax, emit draw y,
// residual draw z, accept bit):
//   y: the draw from p with u(row, emit);
//   z: rows that verify a chain draft with candidates: the draw from
//      (p - q)+ renormalised with the same uniform (y if that is all zero);
//   acc: u(row, accept) * q(x) < p(x) for the row's draft x (q(x) = 0:
//      p(x) > 0).
// Warp 0 applies the policy to the pool while warp 1 builds q, warp 2 draws
// the row's two uniforms and warp 3 reads the draft token.
// q of a draft row, by warp 1: the node's candidates in pool order under the
// request's policy, or the point mass on the draft when no candidates were
// given (a candidate proposed without probabilities, e.g. by an n-gram match)
__device__ __forceinline__ void build_q(const ReqDev& rq, int local, RowShared& rs) {
  const int lane = threadIdx.x & 31;
  if (!rq.q_ids) {
    if (lane == 0) {
      rs.qid[0] = rq.tokens[local];
      rs.qp[0] = 1.0f;
      rs.qm = 1;
    }
    return;
  }
  const float* qv = rq.q_pen + static_cast<size_t>(local) * kQCand;
  const int32_t* qi = rq.q_ids + static_cast<size_t>(local) * kQCand;
  // one load per lane, then ranks by shuffles (no loads inside the loop)
  const int sl = lane < kQCand ? lane : 0;
  const float v = __ldcg(qv + sl);         // possibly penalised earlier in this window
  const int32_t id = qi[sl];
  const uint32_t k = float_key(v);
  int rank = 0;
#pragma unroll
  for (int s2 = 0; s2 < kQCand; ++s2) {
    const uint32_t ks = __shfl_sync(0xffffffffu, k, s2);
    const int32_t is = __shfl_sync(0xffffffffu, id, s2);
    rank += ((ks > k) | ((ks == k) & ((is < id) | ((is == id) & (s2 < lane))))) ? 1 : 0;
  }
  if (lane < kQCand) {
    rs.qid[rank] = id;
    rs.qv[rank] = v;
  }
  __syncwarp();
  policy_warp(rs.qv, kQCand, rq.pol, rs.qe, rs.qpc, &rs.qm, &rs.qS);
  if (lane < rs.qm) rs.qp[lane] = __fdiv_rn(rs.qe[lane], rs.qS);
}

// The parts of a row's decision that need none of the row's logits: the
// chain flag, the draft token, both uniforms and, if with_q, q.  The inputs
// read here were all written before the window's first kernel ran, so the
// row kernel does this before waiting for its predecessor.
__device__ void prepare_row(const ReqDev& rq, int row, bool with_q, RowShared& rs) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (rq.pol.temperature == 0.f) return;
  const int local = row - rq.row0;
  if (tid == 0) rs.chain = 1;
  block_sync();
  if (rq.parent)
    for (int j = tid; j < rq.n_nodes; j += THREADS)
      if (rq.parent[j] != j - 1) rs.chain = 0;
  block_sync();
  // sampled chains take the rejection test: against the draft candidates' q
  // when given, else against q = delta(draft)
  const bool reject_row = rs.chain && local < rq.n_nodes;
  const uint64_t urow = static_cast<uint64_t>(local);
  if (warp == 1 && reject_row && with_q) {
    build_q(rq, local, rs);
  } else if (warp == 2) {
    if (lane == 0) rs.u2 = uniform01(rq.seed, rq.position, urow, kPurposeEmit);
    if (lane == 1 && reject_row) rs.u1 = uniform01(rq.seed, rq.position, urow, kPurposeAccept);
  } else if (warp == 3 && lane == 0 && reject_row) {
    rs.draft = rq.tokens[local];
  }
  block_sync();
}

// The row's decisions (emit draw y, residual draw z, accept bit) once its
// pool is known; prepare_row ran before, and built q.
__device__ void decide_row(const ReqDev& rq, int row, int n, RowShared& rs, int4* dec,
                           bool live = true) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const vr_policy& pol = rq.pol;
  const int local = row - rq.row0;
  if (pol.temperature == 0.f) {
    if (tid == 0) {
      const int4 d = make_int4(rs.ids[0], rs.ids[0], rs.ids[0], 0);
      if (live) dec[row] = d;
      rs.dec = d;
    }
    return;
  }
  const bool reject_row = rs.chain && local < rq.n_nodes;

  if (warp == 0) policy_warp(rs.vals, n, pol, rs.e, rs.pc, &rs.m, &rs.S);
  block_sync();
  if (warp != 0) return;

  const int m = rs.m;
  const float S = rs.S;
  const float u2 = rs.u2;
  const float t2 = __fmul_rn(u2, S);
  int j = warp_first(m, [&](int i) { return rs.pc[i] > t2; });
  if (j < 0) j = last_positive(rs.e, m);
  const int32_t y = rs.ids[j];
  int32_t z = y;
  int acc = 0;
  if (reject_row) {
    const int32_t xd = rs.draft;
    const int qm = rs.qm;
    // residual (p - q)+ over the kept entries; p(x) from the matching entry
    // entries lane and lane + 32 side by side (both divisions in flight)
    float px = 0.0f;
    int32_t qid[kQCand];
    float qp[kQCand];
#pragma unroll
    for (int s2 = 0; s2 < kQCand; ++s2) {
      qid[s2] = s2 < qm ? rs.qid[s2] : -1;
      qp[s2] = s2 < qm ? rs.qp[s2] : 0.0f;
    }
    auto residual_entry = [&](int jj) {
      const int32_t id = rs.ids[jj];
      const float pj = __fdiv_rn(rs.e[jj], S);
      float qj = 0.0f;
#pragma unroll
      for (int s2 = 0; s2 < kQCand; ++s2)
        if (qid[s2] == id) qj = __fadd_rn(qj, qp[s2]);
      const float d = __fsub_rn(pj, qj);
      rs.r[jj] = (jj < m && d > 0.0f) ? d : 0.0f;
      if (jj < m && id == xd) px = pj;
    };
    residual_entry(lane);
    // the upper half only when more than 32 entries are kept (r past m is
    // never read)
    if (m > 32) residual_entry(lane + 32);
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
      rs.acc = (qx > 0.0f) ? (__fmul_rn(rs.u1, qx) < px) : (px > 0.0f);
      running_sums(rs.r, rs.pr, m);
    }
    __syncwarp();
    acc = rs.acc;
    const float sr = rs.pr[m - 1];
    if (sr > 0.0f) {
      const float tz = __fmul_rn(u2, sr);
      int jz = warp_first(m, [&](int i) { return rs.pr[i] > tz; });
      if (jz < 0) jz = last_positive(rs.r, m);
      z = rs.ids[jz];
    }
  }
  if (lane == 0) {
    const int4 d = make_int4(rs.ids[0], y, z, acc);
    if (live) dec[row] = d;
    rs.dec = d;
  }
}

// ---------------------------------------------------------------------------
// acceptance walk of one request (thread 0 writes; the CTA validates)

// The request's tokens and parents into shared memory, checked: bad token,
// bad parent or bad candidate id bits in as.bad, as.not_chain if any node
// does not hang from its predecessor.  Reads inputs only, so the row kernel
// does it before waiting for its predecessor.
__device__ void prepare_accept(const ReqDev& rq, int vocab, AcceptShared& as) {
  const int n = rq.n_nodes, tid = threadIdx.x;
  const bool greedy = rq.pol.temperature == 0.f;
  if (tid == 0) {
    as.bad = 0;
    as.not_chain = 0;
  }
  block_sync();
  if (tid < n) {
    const int t = rq.tokens[tid];
    const int p = rq.parent ? rq.parent[tid] : tid - 1;
    as.tok[tid] = t;
    as.par[tid] = p;
    int b = 0;
    if (t < 0 || t >= vocab) b |= VR_DEV_BAD_TOKEN;
    if (p < -1 || p >= tid) b |= VR_DEV_BAD_PARENT;
    if (p != tid - 1) atomicOr(&as.not_chain, 1);
    if (b) atomicOr(&as.bad, b);
  }
  block_sync();
  const bool rejection = !greedy && !as.not_chain;
  if (rejection && rq.q_ids)
    for (int i = tid; i < n * kQCand; i += THREADS) {
      const int id = rq.q_ids[i];
      if (id < 0 || id >= vocab) atomicOr(&as.bad, VR_DEV_BAD_QID);
    }
  block_sync();
}

// The acceptance walk of one request (warp 0; lane 0 writes), after
// prepare_accept, with every row's decisions in dec.
__device__ void accept_request(const ReqDev& rq, const int4* dec, int32_t* status,
                               AcceptShared& as) {
  const int n = rq.n_nodes, R = n + 1, tid = threadIdx.x, lane = tid & 31;
  const bool greedy = rq.pol.temperature == 0.f;
  const bool rejection = !greedy && !as.not_chain;
  for (int j = tid; j < R; j += THREADS) as.d[j] = __ldcg(dec + rq.row0 + j);
  block_sync();
  if (tid >= 32) return;
  if (!greedy && !rejection && !as.bad) {
    // naive sampling descent: from the root, emit the current row's draw y and
    // move to the lowest-index child of the current node carrying y; one
    // ballot over the (at most 63) nodes finds it
    int32_t* out = rq.out_ids;
    int cur = -1, cnt = 0;
    while (true) {
      const int32_t y = as.d[cur < 0 ? 0 : 1 + cur].y;
      if (lane == 0) out[cnt] = y;
      ++cnt;
      const int j0 = lane, j1 = lane + 32;
      const bool m0 = j0 < n && as.par[j0] == cur && as.tok[j0] == y;
      const bool m1 = j1 < n && as.par[j1] == cur && as.tok[j1] == y;
      const uint32_t b0 = __ballot_sync(0xffffffffu, m0);
      const uint32_t b1 = __ballot_sync(0xffffffffu, m1);
      const int next = b0 ? __ffs(static_cast<int>(b0)) - 1
                          : (b1 ? 32 + __ffs(static_cast<int>(b1)) - 1 : -1);
      if (next < 0) break;
      cur = next;
    }
    if (lane == 0) {
      *rq.out_accept = cnt - 1;
      *rq.out_n = cnt;
    }
    return;
  }
  if (tid != 0) return;
  if (as.bad) {
    set_status(status, as.bad);
    *rq.out_accept = 0;
    *rq.out_n = 0;
    return;
  }
  int32_t* out = rq.out_ids;
  const int4* d = as.d;
  int accepted = 0;
  if (greedy) {
    uint8_t* ok = as.ok;       // in shared memory, not in the thread's local memory
    int32_t* depth = as.depth;
    int best = -1, best_depth = 0;
    for (int j = 0; j < n; ++j) {
      const int p = as.par[j];
      ok[j] = as.tok[j] == d[p < 0 ? 0 : 1 + p].x && (p < 0 || ok[p]);
      depth[j] = p < 0 ? 1 : depth[p] + 1;
      if (ok[j] && depth[j] > best_depth) {
        best = j;
        best_depth = depth[j];
      }
    }
    for (int node = best, k = best_depth - 1; node >= 0; node = as.par[node], --k)
      out[k] = as.tok[node];
    out[best_depth] = d[best < 0 ? 0 : 1 + best].x;
    accepted = best_depth;
  } else if (rejection) {
    int a = 0;
    while (a < n && d[a].w) ++a;
    for (int i = 0; i < a; ++i) out[i] = as.tok[i];
    out[a] = (a < n) ? d[a].z : d[n].y;
    accepted = a;
  }
  *rq.out_accept = accepted;
  *rq.out_n = accepted + 1;
}

// ---------------------------------------------------------------------------
// shared tail of the sampling kernels

struct SampleArgs {
  const float* logits;     // [rows][vocab] (penalised where penalties apply)
  int vocab, seg_len, nseg;
  uint64_t* cand;          // [rows][nseg][64]
  uint32_t* row_ticket;    // [rows], zero between calls
  uint32_t* req_ticket;    // [requests], zero between calls
  unsigned long long* req_mask;  // [requests] chain done/accept bits, zero between calls
  int32_t* pool_ids;       // [rows][out_k]
  float* pool_vals;        // [rows][out_k]
  int out_k;               // leading pool entries written per row (<= 64)
  int4* dec;               // [rows]
  int32_t* status;
  int decide;              // 0: pools only
  float* pen_logits;       // row kernel: penalties applied in place here (== logits), or null
  int warm;                // row kernel: run the instruction warm-up pass before the wait
};

// sh.out[0..count) -> sh.sorted in pool order (zero-padded)
__device__ __forceinline__ void sort_out_into_sorted(SelectShared& sh) {
  const int tid = threadIdx.x;
  if (tid < kPool) {
    uint64_t v = 0ull;
    int rank = tid;
    if (tid < sh.count) {
      v = sh.out[tid];
      rank = 0;
      for (int j = 0; j < sh.count; ++j) rank += (sh.out[j] > v);
    }
    sh.sorted[rank] = v;
  }
  block_sync();
}

// The row's pool (64 composites in pool order, zero-padded) -> pool ids and
// values, then the row's decisions, then (last row of its request) the
// acceptance.  live == false: the row kernel's instruction warm-up pass,
// which writes nothing outside shared memory and stops after the decisions.
__device__ void finish_row(const SampleArgs& a, const ReqTable& tab, int row, const uint64_t* pool,
                           RowShared& rs, AcceptShared& as, int& last, bool prepared,
                           int n_pool = kPool, bool live = true) {
  const int tid = threadIdx.x;
  const float* rp = a.logits + static_cast<size_t>(row) * a.vocab;
  const int n = min(a.vocab, n_pool);
  if (tid < kPool) {
    int32_t id = -1;
    float v = __int_as_float(0x7fffffff);
    // A zero entry is padding (its id decodes to -1).  A pool has fewer than
    // n entries only in the row kernel's warm-up pass, whose group maxima and
    // logits may be mid-rewrite and disagree; such an entry keeps id -1 and a
    // NaN and never reaches the logits reload in value_of_key.
    const uint64_t p = tid < n ? pool[tid] : 0ull;
    if (p != 0ull) {
      id = static_cast<int32_t>(packed_id(p));
      v = value_of_key(static_cast<uint32_t>(p >> 32), rp, id);
    }
    if (live && tid < a.out_k) {
      a.pool_ids[static_cast<size_t>(row) * a.out_k + tid] = id;
      a.pool_vals[static_cast<size_t>(row) * a.out_k + tid] = v;
    }
    rs.ids[tid] = id;
    rs.vals[tid] = v;
  }
  if (!a.decide) return;
  block_sync();
  if (!prepared) load_request(tab, row, rs);
  const ReqDev& rq = rs.req;
  const int b = rs.req_b;
  if (!prepared) prepare_row(rq, row, true, rs);
  decide_row(rq, row, n, rs, a.dec, live);
  if (!live) return;

  // Chains of at most 32 rows: no walk.  Each row writes its own output slot
  // (a draft row: its draft if it accepts it, else its replacement token (the
  // residual draw, or the argmax for greedy requests); the last row: its
  // bonus), then ORs its done bit (1 << local) and its accept bit
  // (<< 32 + local) into the request's word.  The CTA whose OR completes the
  // done bits holds every accept bit in the returned word: the accepted
  // prefix is the leading run of ones, and the slots up to it are already
  // written.  Slots past the emitted ones hold later rows' tokens.
  const int local = row - rq.row0;
  const int R = rq.n_nodes + 1;
  const bool greedy = rq.pol.temperature == 0.f;
  if (a.req_mask && R <= 32 && (!rq.parent || (!greedy && rs.chain))) {
    block_sync();       // rs.dec, written by warp 0
    if (tid == 0) {
      const int4 d = rs.dec;
      int bit = 0;
      int32_t tok = d.y;                         // the last row: its bonus draw
      if (greedy) {
        tok = d.x;                               // the argmax is the draft when it accepts
        bit = local < rq.n_nodes && (prepared ? as.tok[local] : rq.tokens[local]) == d.x;
      } else if (local < rq.n_nodes) {
        bit = d.w;
        tok = bit ? rs.draft : d.z;
      }
      rq.out_ids[local] = tok;
      const unsigned long long mine =
          (1ull << local) | (static_cast<unsigned long long>(bit) << (32 + local));
      const unsigned long long all = atomicOr(&a.req_mask[b], mine) | mine;
      const uint32_t full = R == 32 ? 0xffffffffu : ((1u << R) - 1u);
      last = static_cast<uint32_t>(all) == full;
      rs.acc_bits = static_cast<uint32_t>(all >> 32);
    }
    block_sync();
    if (!last) return;
    if (tid == 0) a.req_mask[b] = 0ull;
    if (!prepared) prepare_accept(rq, a.vocab, as);
    if (tid == 0) {
      if (as.bad) {
        set_status(a.status, as.bad);
        *rq.out_accept = 0;
        *rq.out_n = 0;
      } else {
        const uint32_t rej = ~rs.acc_bits;       // the first row that did not accept
        const int lead = rej ? __ffs(static_cast<int>(rej)) - 1 : 32;
        const int accepted = lead < rq.n_nodes ? lead : rq.n_nodes;
        *rq.out_accept = accepted;
        *rq.out_n = accepted + 1;
      }
    }
    return;
  }

  // the last row of the request to finish walks the request
  __threadfence();
  block_sync();
  if (tid == 0)
    last = atomicAdd(&a.req_ticket[b], 1u) == static_cast<uint32_t>(rq.n_nodes);
  block_sync();
  if (!last) return;
  __threadfence();
  if (tid == 0) a.req_ticket[b] = 0u;
  if (!prepared) prepare_accept(rq, a.vocab, as);
  accept_request(rq, a.dec, a.status, as);
}

// ---------------------------------------------------------------------------
// the kernel


__global__ void __launch_bounds__(THREADS, 2)
    sample_kernel(const __grid_constant__ SampleArgs a, const __grid_constant__ ReqTable tab) {
  extern __shared__ __align__(16) uint8_t dyn_smem[];
  StageShared& st = *reinterpret_cast<StageShared*>(dyn_smem);
  __shared__ RowShared rs;
  __shared__ AcceptShared as;
  __shared__ int last;
  pdl_trigger();
  pdl_wait();
  const int seg = blockIdx.x, row = blockIdx.y, tid = threadIdx.x;
  const float* rp = a.logits + static_cast<size_t>(row) * a.vocab;
  // a plain top-k of at most RM_K entries over at most RM_SEG segments:
  // only each list's first k entries need to be exact, and the lists are
  // merged by ranks
  const bool small_k = !a.decide && a.out_k <= RM_K && a.nseg <= RM_SEG;

  // 1. the segment's top 64, stored in pool order: in one pass when the
  // segment fits the registers (the usual case), else sub-block by sub-block
  {
    SelectShared& sh = st.sel;
    const long long s0 = static_cast<long long>(seg) * a.seg_len;
    const long long s1 = std::min<long long>(s0 + a.seg_len, a.vocab);
    uint64_t carry = 0ull;            // thread t < 64: entry t of the running list
    long long from = s0;
    if (a.seg_len == SEG_FAST && segment_top64_fast(rp, s0, s1, st.fast, small_k ? a.out_k : kPool)) {
      carry = tid < kPool ? st.fast.sorted[tid] : 0ull;
      from = s1;
      block_sync();
    }
    for (long long b = from; b < s1; b += SUB) {
      uint64_t x[ITEMS];
      float f[SUB / THREADS];
#pragma unroll
      for (int i = 0; i < SUB / THREADS; ++i) {
        const long long e = b + i * THREADS + tid;
        f[i] = __ldcg(rp + (e < s1 ? e : b));         // unconditional: loads overlap
      }
#pragma unroll
      for (int i = 0; i < SUB / THREADS; ++i) {
        const long long e = b + i * THREADS + tid;
        x[i] = (e < s1) ? pack_key_id(float_key(f[i]), static_cast<uint32_t>(e)) : 0ull;
      }
      x[ITEMS - 1] = carry;
      if (!block_top64_filtered(x, sh)) {
        block_top64(x, sh);
        sort_out_into_sorted(sh);
      }
      carry = (tid < kPool) ? sh.sorted[tid] : 0ull;
      block_sync();
    }
    if (tid < kPool) a.cand[(static_cast<size_t>(row) * a.nseg + seg) * kPool + tid] = carry;
  }

  // 2. the last segment of the row to finish builds the pool and decides
  __threadfence();
  block_sync();
  if (tid == 0) last = atomicAdd(&a.row_ticket[row], 1u) == static_cast<uint32_t>(a.nseg - 1);
  block_sync();
  if (!last) return;
  __threadfence();
  if (tid == 0) a.row_ticket[row] = 0u;
  const uint64_t* lists = a.cand + static_cast<size_t>(row) * a.nseg * kPool;
  const uint64_t* pool = small_k ? rank_merge(lists, a.nseg, a.out_k, st.mrg)
                                 : merge_lists(lists, a.nseg, st.mrg);
  finish_row(a, tab, row, pool, rs, as, last, false);
}

// ---------------------------------------------------------------------------
// penalties inside the row kernel ("Speculative decoding on RDNA" §04): the
// same arithmetic as the penalty kernel, for the CTA's own row

// H of target row `local`: the last W tokens of (hist || tokens on the path
// root -> node local - 1), through assemble_history.
// Sets sr.h_len, and sr.h_bad for a parent array that is not topological.
__device__ void build_row_history(const ReqDev& rq, int local, RowsShared& sr) {
  const int len = assemble_history<THREADS>(rq, local - 1, sr.H, sr.par, sr.path, &sr.h_len,
                                            &sr.h_bad);
  if (threadIdx.x == 0) sr.h_len = len < 0 ? 0 : len;
  block_sync();
}

// Everything of the row's penalties that needs no logits, before the wait:
// the distinct in-vocabulary tokens of H with their counts (O(W^2) compares),
// the distinct 32-row groups they touch, and, for a chain node checked
// against this row, its draft candidates penalised with this row's history
// (their logits are an input, and nothing reads the penalised copy before
// this kernel builds q from it).
__device__ void prepare_penalties(const ReqDev& rq, int local, int vocab, RowsShared& sr) {
  const int tid = threadIdx.x;
  const vr_policy& pol = rq.pol;
  const int len = sr.h_len;
  if (tid == 0) {
    sr.n_u = 0;
    sr.n_grp = 0;
  }
  block_sync();
  for (int j = tid; j < len; j += THREADS) {
    const int t = sr.H[j];
    bool first = true;
    int count = 0;
    for (int i = 0; i < len; ++i) {
      if (sr.H[i] == t) {
        ++count;
        if (i < j) first = false;
      }
    }
    if (first && t >= 0 && t < vocab) {
      const int u = atomicAdd(&sr.n_u, 1);
      sr.tok_u[u] = t;
      sr.cnt_u[u] = count;
    }
  }
  block_sync();
  const int n_u = sr.n_u;
  for (int u = tid; u < n_u; u += THREADS) {
    const int g = sr.tok_u[u] >> 5;
    bool first = true;
    for (int v = 0; v < u; ++v) first &= (sr.tok_u[v] >> 5) != g;
    if (first) sr.grp_u[atomicAdd(&sr.n_grp, 1)] = g;
  }
  // the node's draft candidates, penalised with this row's history
  const bool chain_node = rq.q_ids && local < rq.n_nodes &&
                          (!rq.parent || rq.parent[local] == local - 1);
  if (chain_node && tid < kQCand) {
    const int32_t t = rq.q_ids[static_cast<size_t>(local) * kQCand + tid];
    int count = 0;
    for (int i = 0; i < len; ++i) count += (sr.H[i] == t);
    const float x = rq.q_logits_in[static_cast<size_t>(local) * kQCand + tid];
    rq.q_pen[static_cast<size_t>(local) * kQCand + tid] = count ? penalize_value(x, count, pol) : x;
  }
  __threadfence();     // q reaches L2 before build_q reads it there
  block_sync();
}

// After the wait: penalise the CTA's row in place (each distinct token of H
// once, from the list prepare_penalties built), then refresh the maxima of
// the groups the penalties touched.  A warp takes eight groups at a time and
// issues their loads together.
__device__ void apply_penalties(const vr_policy& pol, float* row, int vocab, uint32_t* gmax_row,
                                RowsShared& sr) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_u = sr.n_u, n_grp = sr.n_grp;
  for (int u = tid; u < n_u; u += THREADS) {
    const int t = sr.tok_u[u];
    row[t] = penalize_value(__ldcg(row + t), sr.cnt_u[u], pol);
  }
  __threadfence();     // the rewritten logits reach L2 before anyone reads them there
  block_sync();
  constexpr int NW = THREADS / 32, SB = 8;
  for (int g0 = warp; g0 < n_grp; g0 += NW * SB) {
    float x[SB];
#pragma unroll
    for (int b = 0; b < SB; ++b) {
      const int k = g0 + b * NW;       // the same for every lane of the warp
      const long long v = static_cast<long long>(k < n_grp ? sr.grp_u[k] : 0) * 32 + lane;
      x[b] = __ldcg(row + (v < vocab ? v : 0));     // unconditional: loads overlap
    }
#pragma unroll
    for (int b = 0; b < SB; ++b) {
      const int k = g0 + b * NW;
      if (k >= n_grp) continue;
      const int g = sr.grp_u[k];
      const int v = g * 32 + lane;
      const uint32_t m = __reduce_max_sync(0xffffffffu, v < vocab ? float_key(x[b]) : 0u);
      if (lane == 0) gmax_row[g] = m;
    }
  }
  __threadfence();     // group maxima reach L2 before they are read there
  block_sync();
}

// Sampling stage for rows whose group maxima (largest order key per 32
// vocabulary rows) were recorded by the projection: one CTA per row.
//  (a) the row's 64 groups with the largest maxima (ties: lower group index),
//      tau = the maximum of the 64th: at least 64 entries reach tau, and every
//      entry of the row's top 64 lies in those groups at or above tau (a row
//      of fewer than 64 groups takes all of them with tau = the lowest key);
//  (b) the chosen groups' entries at or above tau (at most 64 x 32) are
//      gathered and their top 64 taken;
//  (c) pool, policy, decisions and acceptance as in sample_kernel.
__global__ void __launch_bounds__(THREADS, 2)
    sample_rows_kernel(const __grid_constant__ SampleArgs args,
                       const __grid_constant__ ReqTable tab, uint32_t* __restrict__ gmax,
                       int ngroups) {
  extern __shared__ __align__(16) uint8_t dyn_smem[];
  RowsShared& sr = *reinterpret_cast<RowsShared*>(dyn_smem);
  SelectShared& sh = sr.sel;
  __shared__ RowShared rs;
  __shared__ AcceptShared as;
  __shared__ int last;
  __shared__ SampleArgs s_args;
  pdl_trigger();
  const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // before the wait: everything of the row's decision that needs no logits
  // (this kernel only runs after the window's first kernel, which triggers
  // its dependents only once its own predecessors are complete).  First the
  // kernel's arguments and the row's request go to shared memory, so that
  // no read of theirs after the wait goes to memory.
  {
    constexpr int W = static_cast<int>(sizeof(SampleArgs) / 4);
    static_assert(sizeof(SampleArgs) % 4 == 0 && W <= 64, "argument copy");
    if (warp == 1) {
      const uint32_t* src = reinterpret_cast<const uint32_t*>(&args);
      uint32_t* dst = reinterpret_cast<uint32_t*>(&s_args);
      const uint32_t w0 = src[lane];
      const uint32_t w1 = lane + 32 < W ? src[lane + 32] : 0u;
      if (lane < W) dst[lane] = w0;
      if (lane + 32 < W) dst[lane + 32] = w1;
    }
  }
  load_request(tab, row, rs);
  const SampleArgs& a = s_args;
  const ReqDev& rq0 = rs.req;
  const bool pen = a.pen_logits && penalties_active(rq0.pol);
  if (pen) {
    build_row_history(rq0, row - rq0.row0, sr);
    prepare_penalties(rq0, row - rq0.row0, a.vocab, sr);
  }
  prepare_row(rq0, row, true, rs);
  prepare_accept(rq0, a.vocab, as);
  const float* rp = a.logits + static_cast<size_t>(row) * a.vocab;
  const uint32_t* gm = gmax + static_cast<size_t>(row) * ngroups;

  // The body below runs twice, as a loop (one copy of its instructions).
  // Pass 0, before the wait, works on the logits and group maxima as they
  // stand (the previous window's, or values being overwritten) and writes
  // nothing outside shared memory: it only brings this code into the SM's
  // instruction cache.  Every phase runs once per launch, so on cold code
  // each waited on instruction fetches (a phase ran up to twice as long as
  // warm).  Pass 1 runs after the wait, on the window's logits.  The host
  // asks for pass 0 (a.warm) only when the kernel's CTAs fit on the SMs the
  // projection leaves free, i.e. when they start long before the wait
  // returns; otherwise they start as the projection ends, and pass 0 would
  // only delay them.
#pragma unroll 1
  for (int pass = a.warm ? 0 : 1; pass < 2; ++pass) {
    const bool live = pass == 1;
    if (live) pdl_wait();
    if (live && pen) {
      if (sr.h_bad && tid == 0) set_status(a.status, VR_DEV_BAD_PARENT);
      apply_penalties(rq0.pol, a.pen_logits + static_cast<size_t>(row) * a.vocab, a.vocab,
                      gmax + static_cast<size_t>(row) * ngroups, sr);
    }

    if (rq0.pol.temperature == 0.f) {
      // a greedy request needs only each row's argmax: the largest key among
      // the group maxima, the lowest group holding it, and the lowest id of
      // that key inside the group (the pool's first entry; no other entry is
      // formed)
      uint64_t best = 0ull;
  #pragma unroll
      for (int i = 0; i < GI_MAX; ++i) {
        const int g = i * THREADS + tid;
        const uint32_t k = __ldcg(gm + (g < ngroups ? g : 0));   // unconditional: loads overlap
        const uint64_t c = g < ngroups ? pack_key_id(k, static_cast<uint32_t>(g)) : 0ull;
        best = c > best ? c : best;
      }
  #pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        const uint64_t other = __shfl_xor_sync(0xffffffffu, best, o);
        best = other > best ? other : best;
      }
      if (lane == 0) sr.pool[1 + warp] = best;
      block_sync();
      if (warp == 0) {
        uint64_t b = lane < THREADS / 32 ? sr.pool[1 + lane] : 0ull;
  #pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
          const uint64_t other = __shfl_xor_sync(0xffffffffu, b, o);
          b = other > b ? other : b;
        }
        const uint32_t key = static_cast<uint32_t>(b >> 32);
        const long long v = static_cast<long long>(packed_id(b)) * 32 + lane;
        const uint32_t kv = float_key(__ldcg(rp + (v < a.vocab ? v : 0)));
        const uint32_t ball = __ballot_sync(0xffffffffu, v < a.vocab && kv == key);
        const long long id = v - lane + (ball ? __ffs(ball) - 1 : 0);
        if (lane == 0) sr.pool[0] = pack_key_id(key, static_cast<uint32_t>(id));
      }
      block_sync();
      finish_row(a, tab, row, sr.pool, rs, as, last, true, 1, live);
      continue;
    }

    // (a) the 64 groups with the largest maxima, as composites
    // (max key << 32) | ~group, and (b) their entries at or above the 64th
    // maximum
    {
      uint32_t gk[GI_MAX];
  #pragma unroll
      for (int i = 0; i < GI_MAX; ++i) {
        const int g = i * THREADS + tid;
        gk[i] = __ldcg(gm + (g < ngroups ? g : 0));     // unconditional: loads overlap
      }
      const uint64_t* chosen = sr.fast.sorted;
      if (!keys_top64(gk, ngroups - tid, static_cast<uint32_t>(tid), sr.fast)) {
        uint64_t x[GI_MAX];
  #pragma unroll
        for (int i = 0; i < GI_MAX; ++i) {
          const int g = i * THREADS + tid;
          x[i] = g < ngroups ? pack_key_id(gk[i], static_cast<uint32_t>(g)) : 0ull;
        }
        block_top64(x, sh);
        sort_out_into_sorted(sh);
        chosen = sh.sorted;
      }
      const int nchosen = ngroups < kPool ? ngroups : kPool;
      // 64 chosen groups hold at least 64 entries at or above the 64th group
      // maximum; with fewer groups every entry of every group is a candidate
      const uint32_t tau =
          ngroups < kPool ? 0u : static_cast<uint32_t>(chosen[nchosen - 1] >> 32);
      if (tid == 0) sr.ccount = 0;
      block_sync();
      // the chosen groups' entries at or above tau; warp w takes groups
      // w, w + 8, ...: all of its loads are issued before any is used
      constexpr int GPW = kPool / (THREADS / 32);     // groups per warp
      float fv[GPW];
  #pragma unroll
      for (int t = 0; t < GPW; ++t) {
        const int j = warp + t * (THREADS / 32);
        const long long v =
            static_cast<long long>(packed_id(chosen[j < nchosen ? j : 0])) * 32 + lane;
        fv[t] = __ldcg(rp + (v < a.vocab ? v : 0));       // unconditional: loads overlap
      }
      uint32_t kv[GPW];
  #pragma unroll
      for (int t = 0; t < GPW; ++t) kv[t] = float_key(fv[t]);
      // one slot reservation per warp for all of its groups
      uint64_t cv[GPW];
      uint32_t ball[GPW];
      int total = 0;
  #pragma unroll
      for (int t = 0; t < GPW; ++t) {
        const int j = warp + t * (THREADS / 32);
        const long long v =
            static_cast<long long>(packed_id(chosen[j < nchosen ? j : 0])) * 32 + lane;
        uint64_t c = 0ull;
        if (j < nchosen && v < a.vocab && kv[t] >= tau)
          c = pack_key_id(kv[t], static_cast<uint32_t>(v));
        cv[t] = c;
        ball[t] = __ballot_sync(0xffffffffu, c != 0ull);
        total += __popc(ball[t]);
      }
      int at = 0;
      if (lane == 0 && total) at = atomicAdd(&sr.ccount, total);
      at = __shfl_sync(0xffffffffu, at, 0);
  #pragma unroll
      for (int t = 0; t < GPW; ++t) {
        if (cv[t] != 0ull) sr.cands[at + __popc(ball[t] & ((1u << lane) - 1u))] = cv[t];
        at += __popc(ball[t]);
      }
      block_sync();
    }

    // (c) their top 64, in pool order
    const int n = sr.ccount;
    uint64_t* pool = sr.pool;
    if (n <= GATHER_MAX) {
      if (tid < kPool) pool[tid] = 0ull;
      block_sync();
      rank_into(sr.cands, n, pool);
      block_sync();
    } else {
      uint64_t x[C_MAX / THREADS];
  #pragma unroll
      for (int i = 0; i < C_MAX / THREADS; ++i) {
        const int k = i * THREADS + tid;
        x[i] = k < n ? sr.cands[k] : 0ull;
      }
      block_top64(x, sh);
      sort_out_into_sorted(sh);
      if (tid < kPool) pool[tid] = sh.sorted[tid];
      block_sync();
    }
    finish_row(a, tab, row, pool, rs, as, last, true, kPool, live);
  }
}

__global__ void policy_kernel(const float* __restrict__ pool_vals, int pool_len, vr_policy pol,
                              int32_t* __restrict__ out_m, float* __restrict__ out_e,
                              float* __restrict__ out_S) {
  __shared__ float vals[kPool];
  __shared__ __align__(16) float e[kPool];
  __shared__ __align__(16) float pc[kPool];
  __shared__ int m;
  __shared__ float S;
  pdl_trigger();
  pdl_wait();
  const int row = blockIdx.x;
  for (int j = threadIdx.x; j < kPool; j += 32) vals[j] = pool_vals[static_cast<size_t>(row) * kPool + j];
  __syncwarp();
  policy_warp(vals, pool_len, pol, e, pc, &m, &S);
  for (int j = threadIdx.x; j < kPool; j += 32) out_e[static_cast<size_t>(row) * kPool + j] = e[j];
  if (threadIdx.x == 0) {
    out_m[row] = m;
    out_S[row] = S;
  }
}

}  // namespace smp

namespace {

// Segment length of a row: SEG_FAST (one pass in registers) while the row
// needs at most MAX_SEG such segments, else the smallest multiple of SUB
// that keeps the row within MAX_SEG segments.
long long segment_length(int vocab) {
  if (static_cast<long long>(vocab) <= static_cast<long long>(smp::MAX_SEG) * smp::SEG_FAST)
    return smp::SEG_FAST;
  const long long per = (static_cast<long long>(vocab) + smp::MAX_SEG - 1) / smp::MAX_SEG;
  return (per + smp::SUB - 1) / smp::SUB * smp::SUB;
}

}  // namespace

int select_segments(int vocab) {
  const long long seg_len = segment_length(vocab);
  return static_cast<int>((vocab + seg_len - 1) / seg_len);
}

size_t select_cand_bytes(int rows, int vocab) {
  return static_cast<size_t>(rows) * select_segments(vocab) * kPool * sizeof(uint64_t);
}

int launch_sample(const float* logits, int rows, int vocab, uint64_t* cand, uint32_t* row_ticket,
                  uint32_t* req_ticket, unsigned long long* req_mask, int32_t* pool_ids,
                  float* pool_vals, const ReqTable* tab, int4* dec, int32_t* status,
                  cudaStream_t stream, int out_k) {
  if (out_k < 1 || out_k > kPool) return VR_ERR_ARG;
  const int nseg = select_segments(vocab);
  smp::SampleArgs a;
  a.logits = logits;
  a.vocab = vocab;
  a.seg_len = static_cast<int>(segment_length(vocab));
  a.nseg = nseg;
  a.cand = cand;
  a.row_ticket = row_ticket;
  a.req_ticket = req_ticket;
  a.req_mask = req_mask;
  a.pool_ids = pool_ids;
  a.pool_vals = pool_vals;
  a.out_k = out_k;
  a.dec = dec;
  a.status = status;
  a.decide = tab ? 1 : 0;
  a.pen_logits = nullptr;
  const size_t smem = sizeof(smp::StageShared);
  static std::atomic<bool> attr_set[kMaxDevices];
  if (set_smem_limit_once(smp::sample_kernel, static_cast<int>(smem), attr_set) != cudaSuccess)
    return VR_ERR_CUDA;
  ReqTable none{};
  return launch_pdl(smp::sample_kernel, dim3(nseg, rows), dim3(smp::THREADS), smem, stream, a,
                    tab ? *tab : none) == cudaSuccess
             ? VR_OK
             : VR_ERR_CUDA;
}

bool sample_rows_supported(int vocab) {
  return (vocab + 31) / 32 <= smp::GI_MAX * smp::THREADS;
}

int launch_sample_rows(const float* logits, int rows, int vocab, uint32_t* gmax,
                       uint32_t* req_ticket, unsigned long long* req_mask, int32_t* pool_ids,
                       float* pool_vals, const ReqTable& tab, int4* dec, int32_t* status,
                       float* pen_logits, bool warm, cudaStream_t stream) {
  smp::SampleArgs a{};
  a.logits = logits;
  a.vocab = vocab;
  a.req_ticket = req_ticket;
  a.req_mask = req_mask;
  a.pool_ids = pool_ids;
  a.pool_vals = pool_vals;
  a.out_k = kPool;
  a.dec = dec;
  a.status = status;
  a.decide = 1;
  a.pen_logits = pen_logits;
  a.warm = warm ? 1 : 0;
  const size_t smem = sizeof(smp::RowsShared);
  static std::atomic<bool> attr_set[kMaxDevices];
  if (set_smem_limit_once(smp::sample_rows_kernel, static_cast<int>(smem), attr_set) != cudaSuccess)
    return VR_ERR_CUDA;
  return launch_pdl(smp::sample_rows_kernel, dim3(rows), dim3(smp::THREADS), smem, stream, a, tab,
                    gmax, (vocab + 31) / 32) == cudaSuccess
             ? VR_OK
             : VR_ERR_CUDA;
}

int launch_policy(const float* pool_vals, int rows, int pool_len, const vr_policy& pol,
                  int32_t* out_m, float* out_e, float* out_S, cudaStream_t stream) {
  return launch_pdl(smp::policy_kernel, dim3(rows), dim3(32), 0, stream, pool_vals, pool_len, pol,
                    out_m, out_e, out_S) == cudaSuccess
             ? VR_OK
             : VR_ERR_CUDA;
}

}  // namespace vr
