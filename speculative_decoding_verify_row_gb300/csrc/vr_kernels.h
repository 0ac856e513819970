// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "vr_common.cuh"

namespace vr {

// Per-device host state.  A kernel's dynamic shared-memory limit and the SM
// count belong to a device, not to the process, so the launchers remember
// them per device ordinal.  Two threads may both fill one entry; they store
// the same value.
constexpr int kMaxDevices = 64;

// cudaFuncSetAttribute(kernel, MaxDynamicSharedMemorySize, bytes) on the
// current device, once per device; `done` is the kernel's own flag array.
// Devices past kMaxDevices get the call on every launch.
template <class K>
inline cudaError_t set_smem_limit_once(K kernel, int bytes,
                                       std::atomic<bool> (&done)[kMaxDevices]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cached = dev >= 0 && dev < kMaxDevices;
  if (cached && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && cached) done[dev].store(true, std::memory_order_release);
  return e;
}

// SM count of the current device (looked up once per device); 0 on failure.
inline int device_sm_count() {
  static std::atomic<int> sms[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < kMaxDevices) {
    const int n = sms[dev].load(std::memory_order_acquire);
    if (n > 0) return n;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < kMaxDevices) sms[dev].store(n, std::memory_order_release);
  return n;
}

// host inputs -> workspace by a kernel that reads device-mapped pinned host
// memory (src: device addresses of pinned host buffers; dst: workspace)
constexpr int kMaxStageSegs = 6;
struct StageSeg {
  const uint32_t* src;
  uint32_t* dst;
  uint32_t words;
};
int launch_stage_inputs(const StageSeg* segs, int nseg, cudaStream_t stream);
// The request table of a batched window into the workspace (table[n_req],
// row_req[rows]) by kernels that carry it in their parameters, 128 requests
// per launch: nothing on the stream reads host memory of the call.
int launch_stage_requests(const ReqDev* reqs, int n_req, ReqDev* table, int32_t* row_req,
                          cudaStream_t stream);

// projection
bool encode_bf16_tile(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                      uint32_t box_inner, uint32_t box_outer);
bool encode_f32_box_sw128(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                          uint32_t box_inner, uint32_t box_outer);
size_t tcb_plane_bytes(int rows, int hidden);
// gmax (nullable): [rows][ceil(vocab/32)] largest order key per 32 vocab rows
// logits2 (nullable): a second buffer receiving the same logits
int launch_project_tcb(const uint16_t* weight, const float* act, int rows, int hidden, int vocab,
                       float* logits, float* logits2, void* planes, uint32_t* gmax,
                       int32_t* status, cudaStream_t stream);
// scratch (tc_scratch_bytes, 16-byte aligned): the activation planes for
// more than 16 rows, else room for an aligned copy of act
size_t tc_scratch_bytes(int rows, int hidden);
// SMs that the tensor-core projection of `rows` rows leaves free, at its
// start or at least one unit of work before its end (its grid may leave room
// for the row sampling kernel that follows it in a window, and CTAs with one
// unit fewer than the others end early)
int tc_early_free_sms(int rows, int vocab);
int launch_project_tc(const uint16_t* weight, const float* act, int rows, int hidden, int vocab,
                      float* logits, float* logits2, void* scratch, uint32_t* gmax,
                      int32_t* status, cudaStream_t stream);
int ffma_rows_per_pass(int hidden);
int launch_project_ffma(const uint16_t* weight, const float* act, int rows, int hidden, int vocab,
                        float* logits, cudaStream_t stream);

// penalties: rows_total rows of `logits` (stride vocab), requests in `tab`
int launch_penalize(const ReqTable& tab, int rows_total, float* logits, int vocab,
                    bool with_q, int32_t* status, cudaStream_t stream);

// sampling stage, one kernel: logits [rows][vocab] -> pool ids/vals
// [rows][64]; with a request table also the policy, the per-row decisions
// dec[row] = (argmax, emit draw y, residual draw z, accept bit) and the
// acceptance of every request (a walk over the rows' decisions, or for
// chains of at most 32 rows the per-request done/accept bits in req_mask).
// row_ticket [rows], req_ticket and req_mask [requests] must be zero on
// entry and are zero again on exit.
int select_segments(int vocab);
size_t select_cand_bytes(int rows, int vocab);
// out_k: entries written per row to pool_ids/pool_vals (row stride out_k);
// the decisions always use the whole 64-wide pool.
int launch_sample(const float* logits, int rows, int vocab, uint64_t* cand, uint32_t* row_ticket,
                  uint32_t* req_ticket, unsigned long long* req_mask, int32_t* pool_ids,
                  float* pool_vals, const ReqTable* tab,
                  int4* dec, int32_t* status, cudaStream_t stream, int out_k = kPool);

// the same stage for rows whose group maxima gmax [rows][ceil(vocab/32)]
// (largest order key per 32 vocabulary rows) are known: one CTA per row
bool sample_rows_supported(int vocab);
// warm: the kernel's CTAs start well before its wait returns (they fit beside
// the projection), so it first runs its body once without effect to load its
// instructions.  pen_logits (== logits, or null): the kernel applies each
// active request's penalties to its own rows there first (and refreshes
// gmax), so no penalty kernel runs before it; the counts, and the penalised
// draft candidates, are prepared before its wait.
int launch_sample_rows(const float* logits, int rows, int vocab, uint32_t* gmax,
                       uint32_t* req_ticket, unsigned long long* req_mask, int32_t* pool_ids,
                       float* pool_vals,
                       const ReqTable& tab, int4* dec, int32_t* status, float* pen_logits,
                       bool warm, cudaStream_t stream);

int launch_policy(const float* pool_vals, int rows, int pool_len, const vr_policy& pol,
                  int32_t* out_m, float* out_e, float* out_S, cudaStream_t stream);

}  // namespace vr
