// Acceptance of one verify window per CTA.
//
//   greedy chain / tree  -- "Speculative decoding on RDNA" §02 and the §01
//     figure (longest argmax-matching prefix, then the argmax at the first
//     mismatch or the bonus); trees: the deepest node whose whole path
//     agrees with the argmax of each parent row ("One RDNA4 verify pass
//     ...", "Spend the budget on a tree"), equal depths to the lower index.
//   sampled chain with draft candidates -- rejection sampling (§03 steps
//     1-4): the first rejected draft ends the window with its residual
//     draw; after k acceptances the bonus draw of row k.
//   sampled tree, or sampled chain without candidates -- naive sampling
//     descent ("feat(dflash) ...": exact for a deterministic draft).
//
// Every random decision belongs to one row and has already been taken by
// that row's select CTA (dec[row] = argmax, emit draw, residual draw,
// accept bit).  What is left is to validate the request's device data and
// walk its rows with integer compares.
#include "vr_common.cuh"
#include "vr_kernels.h"

namespace vr {
namespace acc {

constexpr int THREADS = 64;
constexpr int MAXR = VR_MAX_WINDOW_ROWS;

__global__ void __launch_bounds__(THREADS)
    accept_kernel(ReqTable tab, int vocab, const int4* __restrict__ dec, int32_t* status) {
  __shared__ int32_t tok[MAXR], par[MAXR];
  __shared__ int4 d[MAXR];
  __shared__ int bad, not_chain;

  const ReqDev& rq = request(tab, blockIdx.x);
  const int n = rq.n_nodes, R = n + 1;
  const int tid = threadIdx.x;
  const bool greedy = rq.pol.temperature == 0.f;

  if (tid == 0) {
    bad = 0;
    not_chain = 0;
  }
  __syncthreads();
  for (int j = tid; j < R; j += THREADS) d[j] = dec[rq.row0 + j];
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
  if (rejection)
    for (int i = tid; i < n * kQCand; i += THREADS) {
      const int id = rq.q_ids[i];
      if (id < 0 || id >= vocab) atomicOr(&bad, VR_DEV_BAD_QID);
    }
  __syncthreads();
  if (tid != 0) return;
  if (bad) {
    set_status(status, bad);
    *rq.out_accept = 0;
    *rq.out_n = 0;
    return;
  }
  int32_t* out = rq.out_ids;
  int accepted = 0;
  if (greedy) {
    bool ok[MAXR];
    int depth[MAXR];
    int best = -1, best_depth = 0;
    for (int j = 0; j < n; ++j) {
      const int p = par[j];
      ok[j] = tok[j] == d[p < 0 ? 0 : 1 + p].x && (p < 0 || ok[p]);
      depth[j] = p < 0 ? 1 : depth[p] + 1;
      if (ok[j] && depth[j] > best_depth) {
        best = j;
        best_depth = depth[j];
      }
    }
    for (int node = best, k = best_depth - 1; node >= 0; node = par[node], --k) out[k] = tok[node];
    out[best_depth] = d[best < 0 ? 0 : 1 + best].x;
    accepted = best_depth;
  } else if (rejection) {
    int a = 0;
    while (a < n && d[a].w) ++a;
    for (int i = 0; i < a; ++i) out[i] = tok[i];
    out[a] = (a < n) ? d[a].z : d[n].y;
    accepted = a;
  } else {
    int cur = -1, cnt = 0;
    while (true) {
      const int32_t y = d[cur < 0 ? 0 : 1 + cur].y;
      out[cnt++] = y;
      int next = -1;
      for (int j = cur + 1; j < n; ++j)
        if (par[j] == cur && tok[j] == y) {
          next = j;
          break;
        }
      if (next < 0) break;
      cur = next;
    }
    accepted = cnt - 1;
  }
  *rq.out_accept = accepted;
  *rq.out_n = accepted + 1;
}

}  // namespace acc

int launch_accept(const ReqTable& tab, int n_req, int vocab, const int4* dec, int32_t* status,
                  cudaStream_t stream) {
  acc::accept_kernel<<<n_req, acc::THREADS, 0, stream>>>(tab, vocab, dec, status);
  return cudaGetLastError() == cudaSuccess ? VR_OK : VR_ERR_CUDA;
}

}  // namespace vr
