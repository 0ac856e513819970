// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "vr_common.cuh"

namespace vr {

// projection
size_t tc_plane_bytes(int rows, int hidden);
int launch_project_tc(const uint16_t* weight, const float* act, int rows, int hidden, int vocab,
                      float* logits, void* planes, int32_t* status, cudaStream_t stream);
int ffma_rows_per_pass(int hidden);
int launch_project_ffma(const uint16_t* weight, const float* act, int rows, int hidden, int vocab,
                        float* logits, cudaStream_t stream);

// penalties: rows_total rows of `logits` (stride vocab), requests in `tab`
int launch_penalize(const ReqTable& tab, int rows_total, float* logits, int vocab,
                    bool with_q, int32_t* status, cudaStream_t stream);

// pool select (+ optional policy): logits [rows][vocab] ->
// pool ids/vals [rows][64], and if tab != nullptr e/m/S per row
int select_segments(int vocab);
size_t select_cand_bytes(int rows, int vocab);
int launch_select(const float* logits, int rows, int vocab, uint64_t* cand, int32_t* pool_ids,
                  float* pool_vals, const ReqTable* tab, double* pol_e, int32_t* pol_m,
                  double* pol_S, cudaStream_t stream);

int launch_policy(const float* pool_vals, int rows, int pool_len, const vr_policy& pol,
                  int32_t* out_m, double* out_e, double* out_S, cudaStream_t stream);

// acceptance: one CTA per request
int launch_accept(const ReqTable& tab, int n_req, int vocab, const int32_t* pool_ids,
                  const double* pol_e, const int32_t* pol_m, const double* pol_S,
                  const float* q_pen, int32_t* status, cudaStream_t stream);

}  // namespace vr
