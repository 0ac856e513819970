// Staging of a window's host inputs by a kernel, for the host-buffer entry
// points: the inputs live in pinned (page-locked, device-mapped) host memory
// and are read by the GPU directly, before the kernel waits for its
// predecessor, so the host-link latency overlaps the previous window; after
// the wait the words are stored into the workspace.  This replaces one
// host-to-device copy per input, each of which would serialise on the stream
// and keep the projection from launching early.
#include "vr_common.cuh"
#include "vr_kernels.h"

namespace vr {
namespace {

constexpr int kStageThreads = 256;
constexpr int kStagePerThread = 4;      // words held in registers per thread

struct StageArgs {
  StageSeg seg[kMaxStageSegs];
  uint32_t end[kMaxStageSegs];          // running word counts
  int nseg;
};

__device__ __forceinline__ int seg_of(const StageArgs& a, uint32_t w) {
  int s = 0;
  while (s + 1 < a.nseg && w >= a.end[s]) ++s;
  return s;
}

__global__ void __launch_bounds__(kStageThreads)
    stage_inputs_kernel(const __grid_constant__ StageArgs a) {
  // The kernel that follows (a projection or its split pass) reads nothing
  // of the window before its own wait, only the weights, so it may launch
  // at once and start its weight stream while the previous window ends.
  // The kernels after it launch only once it is past its wait, by which
  // time this kernel has completed.
  pdl_trigger();
  const uint32_t total = a.end[a.nseg - 1];
  const uint32_t base = blockIdx.x * (kStageThreads * kStagePerThread) + threadIdx.x;
  uint32_t v[kStagePerThread];
  // host reads first: nothing before this kernel writes the host buffers
#pragma unroll
  for (int i = 0; i < kStagePerThread; ++i) {
    const uint32_t w = base + i * kStageThreads;
    v[i] = 0u;
    if (w < total) {
      const int s = seg_of(a, w);
      const uint32_t off = w - (s ? a.end[s - 1] : 0u);
      v[i] = a.seg[s].src[off];
    }
  }
  // the workspace may still be read by the previous window's kernels
  pdl_wait();
#pragma unroll
  for (int i = 0; i < kStagePerThread; ++i) {
    const uint32_t w = base + i * kStageThreads;
    if (w < total) {
      const int s = seg_of(a, w);
      const uint32_t off = w - (s ? a.end[s - 1] : 0u);
      a.seg[s].dst[off] = v[i];
    }
  }
}

// The request table of a batched window, passed by value and stored into
// the workspace with the row-to-request map, one CTA per chunk of requests.
// Kernel parameters are copied when the launch is made (or captured into a
// graph), so the table needs no host buffer that outlives the call; a copy
// from the call's own host memory would, in a captured graph, read that
// memory again at every replay, long after the call returned.
constexpr int kReqChunk = 128;           // 128 x 136 B of requests: within the parameter space

struct ReqChunk {
  ReqDev r[kReqChunk];
  int n;                                 // requests in this chunk
  int b0;                                // index of its first request
};

__global__ void __launch_bounds__(kStageThreads)
    stage_requests_kernel(const __grid_constant__ ReqChunk c, ReqDev* __restrict__ table,
                          int32_t* __restrict__ row_req) {
  // as for the inputs: the projection after this kernel reads only weights
  // before its wait, and the row kernel launches only after that wait
  pdl_trigger();
  // the table and the map may still be read by the previous window's kernels
  pdl_wait();
  constexpr int W = static_cast<int>(sizeof(ReqDev) / 4);
  static_assert(sizeof(ReqDev) % 4 == 0, "request copy");
  const uint32_t* src = reinterpret_cast<const uint32_t*>(c.r);
  uint32_t* dst = reinterpret_cast<uint32_t*>(table + c.b0);
  for (int w = threadIdx.x; w < c.n * W; w += kStageThreads) dst[w] = src[w];
  for (int i = threadIdx.x >> 5; i < c.n; i += kStageThreads / 32) {
    const ReqDev& q = c.r[i];
    for (int j = threadIdx.x & 31; j <= q.n_nodes; j += 32) row_req[q.row0 + j] = c.b0 + i;
  }
}

}  // namespace

int launch_stage_inputs(const StageSeg* segs, int nseg, cudaStream_t stream) {
  if (nseg < 1 || nseg > kMaxStageSegs) return VR_ERR_ARG;
  StageArgs a{};
  uint64_t total = 0;
  int n = 0;
  for (int i = 0; i < nseg; ++i) {
    if (segs[i].words == 0) continue;
    total += segs[i].words;
    a.seg[n] = segs[i];
    a.end[n] = static_cast<uint32_t>(total);
    ++n;
  }
  if (n == 0) return VR_OK;
  if (total > 0xffffffffull - kStageThreads * kStagePerThread) return VR_ERR_ARG;
  a.nseg = n;
  const uint32_t per_cta = kStageThreads * kStagePerThread;
  const uint32_t grid = static_cast<uint32_t>((total + per_cta - 1) / per_cta);
  return launch_pdl(stage_inputs_kernel, dim3(grid), dim3(kStageThreads), 0, stream, a) ==
                 cudaSuccess
             ? VR_OK
             : VR_ERR_CUDA;
}

int launch_stage_requests(const ReqDev* reqs, int n_req, ReqDev* table, int32_t* row_req,
                          cudaStream_t stream) {
  static_assert(sizeof(ReqChunk) <= 32000, "kernel parameter space");
  for (int b0 = 0; b0 < n_req; b0 += kReqChunk) {
    ReqChunk c;
    c.n = n_req - b0 < kReqChunk ? n_req - b0 : kReqChunk;
    c.b0 = b0;
    for (int i = 0; i < c.n; ++i) c.r[i] = reqs[b0 + i];
    if (launch_pdl(stage_requests_kernel, dim3(1), dim3(kStageThreads), 0, stream, c, table,
                   row_req) != cudaSuccess)
      return VR_ERR_CUDA;
  }
  return VR_OK;
}

}  // namespace vr
