// Acceptance of one verify window per CTA.
//
//   greedy chain / tree  -- "Speculative decoding on RDNA" §02 and the §01
//     figure (longest argmax-matching prefix, then the argmax at the first
//     mismatch or the bonus); trees: the deepest node whose whole path
//     agrees with the argmax of each parent row ("One RDNA4 verify pass
//     ...", "Spend the budget on a tree"), equal depths to the lower index.
//   sampled chain with draft candidates -- rejection sampling (§03 steps
//     1-4): accept d_i iff u1 * q_i(d_i) < p_i(d_i); on rejection a draw
//     from (p_i - q_i)+ renormalised; after k acceptances the bonus from p_k.
//   sampled tree, or sampled chain without candidates -- naive sampling
//     descent ("feat(dflash) ...": exact for a deterministic draft).
//
// Every random decision of a row depends only on that row (its pool, its
// policy weights, its q and its own Philox uniforms), so all of them are
// computed in parallel, one thread per row; thread 0 then only walks the
// rows with integer compares.  Sums stay sequential in pool order inside
// each row, as the policy defines them.
#include "vr_common.cuh"
#include "vr_kernels.h"

namespace vr {
namespace acc {

constexpr int THREADS = 256;
constexpr int MAXR = VR_MAX_WINDOW_ROWS;

__global__ void __launch_bounds__(THREADS)
    accept_kernel(ReqTable tab, int vocab, const int32_t* __restrict__ pool_ids,
                  const double* __restrict__ pol_e, const int32_t* __restrict__ pol_m,
                  const double* __restrict__ pol_S, int32_t* status) {
  __shared__ int32_t tok[MAXR], par[MAXR];
  __shared__ int32_t argmax[MAXR], y[MAXR], z[MAXR];
  __shared__ int accepted[MAXR];
  __shared__ int32_t qid[MAXR][kQCand];
  __shared__ double qe[MAXR][kQCand];
  __shared__ int qm[MAXR];
  __shared__ double qS[MAXR];
  __shared__ float qv_sorted[THREADS / 32][kQCand];
  __shared__ double e_scratch[THREADS / 32][kPool];
  __shared__ int bad, not_chain;

  const ReqDev& rq = request(tab, blockIdx.x);
  const int n = rq.n_nodes, R = n + 1, base = rq.row0;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const vr_policy& pol = rq.pol;
  const bool greedy = pol.temperature == 0.f;

  if (tid == 0) {
    bad = 0;
    not_chain = 0;
  }
  __syncthreads();
  if (tid < n) {
    const int t = rq.tokens[tid];
    const int p = rq.parent ? rq.parent[tid] : tid - 1;
    tok[tid] = t;
    par[tid] = p;
    int b = 0;
    if (t < 0 || t >= vocab) b |= VR_DEV_BAD_TOKEN;
    if (p < -1 || p >= tid) b |= VR_DEV_BAD_PARENT;
    if (p != tid - 1) atomicOr(&not_chain, 1);
    if (b) atomicOr(&bad, b);
  }
  __syncthreads();
  const bool rejection = !greedy && rq.q_ids != nullptr && !not_chain;
  if (rejection) {
    for (int i = tid; i < n * kQCand; i += THREADS) {
      const int id = rq.q_ids[i];
      if (id < 0 || id >= vocab) atomicOr(&bad, VR_DEV_BAD_QID);
    }
  }
  __syncthreads();
  if (bad) {
    if (tid == 0) {
      set_status(status, bad);
      *rq.out_accept = 0;
      *rq.out_n = 0;
    }
    return;
  }

  // q_i: the draft's 8 candidates in pool order, then the same policy
  if (rejection) {
    for (int j = warp; j < n; j += THREADS / 32) {
      const float* qv = rq.q_pen + static_cast<size_t>(j) * kQCand;
      const int32_t* qi = rq.q_ids + static_cast<size_t>(j) * kQCand;
      if (lane < kQCand) {
        const uint32_t k = float_key(qv[lane]);
        const int32_t id = qi[lane];
        int rank = 0;
        for (int s = 0; s < kQCand; ++s) {
          const uint32_t ks = float_key(qv[s]);
          const int32_t is = qi[s];
          rank += (ks > k) || (ks == k && (is < id || (is == id && s < lane)));
        }
        qid[j][rank] = id;
        qv_sorted[warp][rank] = qv[lane];
      }
      __syncwarp();
      int m;
      double S;
      __shared__ int m_w[THREADS / 32];
      __shared__ double S_w[THREADS / 32];
      policy_warp(qv_sorted[warp], kQCand, pol, e_scratch[warp], &m_w[warp], &S_w[warp]);
      m = m_w[warp];
      S = S_w[warp];
      if (lane < kQCand) qe[j][lane] = e_scratch[warp][lane];
      if (lane == 0) {
        qm[j] = m;
        qS[j] = S;
      }
      __syncwarp();
    }
  }
  __syncthreads();

  // per-row decisions
  if (tid < R) {
    const int row = base + tid;
    const int32_t* ids = pool_ids + static_cast<size_t>(row) * kPool;
    argmax[tid] = ids[0];
    if (!greedy) {
      const double* e = pol_e + static_cast<size_t>(row) * kPool;
      const int m = pol_m[row];
      const double S = pol_S[row];
      const double u2 = uniform01(rq.seed, rq.position, static_cast<uint64_t>(tid), kPurposeEmit);
      const int yj = draw_index(e, m, S, u2);
      y[tid] = ids[yj];
      if (rejection && tid < n) {
        const int32_t x = tok[tid];
        const double px = prob_of(ids, e, m, S, x);
        const double qx = prob_of(qid[tid], qe[tid], qm[tid], qS[tid], x);
        const double u1 =
            uniform01(rq.seed, rq.position, static_cast<uint64_t>(tid), kPurposeAccept);
        accepted[tid] = (qx > 0.0) ? (__dmul_rn(u1, qx) < px) : (px > 0.0);
        // residual (p - q)+ over the kept target entries, in pool order
        double sr = 0.0;
        for (int j = 0; j < m; ++j) {
          double d = __dsub_rn(__ddiv_rn(e[j], S), prob_of(qid[tid], qe[tid], qm[tid], qS[tid], ids[j]));
          sr = __dadd_rn(sr, d > 0.0 ? d : 0.0);
        }
        if (sr > 0.0) {
          const double t = __dmul_rn(u2, sr);
          double c = 0.0;
          int pick = -1, last_pos = 0;
          for (int j = 0; j < m; ++j) {
            double d = __dsub_rn(__ddiv_rn(e[j], S), prob_of(qid[tid], qe[tid], qm[tid], qS[tid], ids[j]));
            d = d > 0.0 ? d : 0.0;
            if (d > 0.0) last_pos = j;
            c = __dadd_rn(c, d);
            if (pick < 0 && c > t) pick = j;
          }
          z[tid] = ids[pick >= 0 ? pick : last_pos];
        } else {
          z[tid] = y[tid];
        }
      }
    }
  }
  __syncthreads();

  if (tid == 0) {
    int32_t* out = rq.out_ids;
    int accepted_n = 0;
    if (greedy) {
      bool ok[MAXR];
      int depth[MAXR];
      int best = -1, best_depth = 0;
      for (int j = 0; j < n; ++j) {
        const int p = par[j];
        ok[j] = tok[j] == argmax[p < 0 ? 0 : 1 + p] && (p < 0 || ok[p]);
        depth[j] = p < 0 ? 1 : depth[p] + 1;
        if (ok[j] && depth[j] > best_depth) {
          best = j;
          best_depth = depth[j];
        }
      }
      for (int node = best, d = best_depth - 1; node >= 0; node = par[node], --d) out[d] = tok[node];
      out[best_depth] = argmax[best < 0 ? 0 : 1 + best];
      accepted_n = best_depth;
    } else if (rejection) {
      int a = 0;
      while (a < n && accepted[a]) ++a;
      for (int i = 0; i < a; ++i) out[i] = tok[i];
      out[a] = (a < n) ? z[a] : y[n];
      accepted_n = a;
    } else {
      int cur = -1, cnt = 0;
      while (true) {
        const int32_t yv = y[cur < 0 ? 0 : 1 + cur];
        out[cnt++] = yv;
        int next = -1;
        for (int j = cur + 1; j < n; ++j)
          if (par[j] == cur && tok[j] == yv) {
            next = j;
            break;
          }
        if (next < 0) break;
        cur = next;
      }
      accepted_n = cnt - 1;
    }
    *rq.out_accept = accepted_n;
    *rq.out_n = accepted_n + 1;
  }
}

}  // namespace acc

int launch_accept(const ReqTable& tab, int n_req, int vocab, const int32_t* pool_ids,
                  const double* pol_e, const int32_t* pol_m, const double* pol_S,
                  const float* /*q_pen*/, int32_t* status, cudaStream_t stream) {
  acc::accept_kernel<<<n_req, acc::THREADS, 0, stream>>>(tab, vocab, pool_ids, pol_e, pol_m, pol_S,
                                                         status);
  return cudaGetLastError() == cudaSuccess ? VR_OK : VR_ERR_CUDA;
}

}  // namespace vr
