// Per-row penalty prepass ("Speculative decoding on RDNA" §04).
//
// Row r of a request is penalised against H_r = the last W tokens of
// (hist || tokens on the path root -> node r-1): for a chain that is
// (prompt || emitted || drafts[0..r)).  A draft node j's candidate logits
// (q) use the history of the row that node is checked against,
// row(parent[j]), so p and q are penalised by the same H (same section).
//
// One CTA per target row and one per draft node: the CTA assembles H in
// shared memory (assemble_history), each thread takes one history slot,
// counts that token's
// occurrences and, if the slot is the token's first occurrence, rewrites
// the logit once.  Distinct tokens never touch the same element, so the
// scattered writes need no ordering.  Cost: O(W^2) compares per row with
// W <= 512 and at most W writes per row.
#include "vr_common.cuh"
#include "vr_kernels.h"

namespace vr {
namespace pen {

constexpr int THREADS = 128;

__global__ void __launch_bounds__(THREADS)
    penalize_kernel(const __grid_constant__ ReqTable tab, int rows_total, float* __restrict__ logits, int vocab,
                    int with_q, int32_t* status) {
  __shared__ int32_t H[VR_MAX_PENALTY_WINDOW];
  __shared__ int32_t par[VR_MAX_WINDOW_ROWS];
  __shared__ int32_t path[VR_MAX_WINDOW_ROWS];
  __shared__ int path_len, bad;

  pdl_trigger();
  pdl_wait();
  const bool is_q = blockIdx.x >= static_cast<unsigned>(rows_total);
  const int g_row = is_q ? blockIdx.x - rows_total : blockIdx.x;   // global row
  const int g = g_row;
  const ReqDev& rq = request(tab, request_of_row(tab, g));
  const vr_policy& pol = rq.pol;
  const int local = g - rq.row0;
  if (!penalties_active(pol)) return;
  if (is_q && (!with_q || !rq.q_ids || local >= rq.n_nodes)) return;

  // the node whose path ends the history: target row r -> node r-1;
  // draft node j -> parent[j]
  int end_node;
  if (!is_q) {
    end_node = local - 1;
  } else {
    end_node = rq.parent ? rq.parent[local] : local - 1;
  }

  int len = assemble_history<THREADS>(rq, end_node, H, par, path, &path_len, &bad);
  if (len < 0) {
    if (threadIdx.x == 0) set_status(status, VR_DEV_BAD_PARENT);
    len = 0;
  }

  if (!is_q) {
    float* row = logits + static_cast<size_t>(g) * vocab;
    for (int j = threadIdx.x; j < len; j += THREADS) {
      const int t = H[j];
      bool first = true;
      int count = 0;
      for (int i = 0; i < len; ++i) {
        if (H[i] == t) {
          ++count;
          if (i < j) first = false;
        }
      }
      if (first && t >= 0 && t < vocab) row[t] = penalize_value(__ldcg(row + t), count, pol);
    }
  } else {
    // candidates of node `local`, written to the request's q buffer
    const int32_t* ids = rq.q_ids + static_cast<size_t>(local) * kQCand;
    const float* in = rq.q_logits_in + static_cast<size_t>(local) * kQCand;
    float* out = rq.q_pen + static_cast<size_t>(local) * kQCand;
    if (threadIdx.x < kQCand) {
      const int t = ids[threadIdx.x];
      int count = 0;
      for (int i = 0; i < len; ++i) count += (H[i] == t);
      const float x = __ldcg(in + threadIdx.x);
      out[threadIdx.x] = count ? penalize_value(x, count, pol) : x;
    }
  }
}

}  // namespace pen

// A request's q copy in the workspace exists only when its penalties are
// active, and then the q blocks write all 8 candidates (penalised or not),
// so no separate copy pass is needed.
int launch_penalize(const ReqTable& tab, int rows_total, float* logits, int vocab, bool with_q,
                    int32_t* status, cudaStream_t stream) {
  const int blocks = rows_total * (with_q ? 2 : 1);
  return launch_pdl(pen::penalize_kernel, dim3(blocks), dim3(pen::THREADS), 0, stream, tab,
                    rows_total, logits, vocab, with_q ? 1 : 0, status) == cudaSuccess
             ? VR_OK
             : VR_ERR_CUDA;
}

}  // namespace vr
