// Verify projection on the CUDA cores: a multi-row GEMV with fp32 FMAs.
//
//   logits[r][v] = sum_h W[v][h] * A[r][h]
//
// "Speculative decoding on RDNA" §02: a row's sum inside a multi-row verify
// projection follows the order of the one-row projection.  Here each (r, v) is summed the same way
// whatever the row count: lane l of a warp owns the 8-wide hidden chunks
// l, l+32, l+64, ... and accumulates them in that order with one FMA per
// element (h ascending inside a chunk); the 32 lane sums are then combined
// by the xor-butterfly 16, 8, 4, 2, 1.  Rows are processed in passes of up
// to RB (<= 8) rows; a pass's rows share every weight load, and the packed
// FFMA2 instruction pairs two vocab rows, each half being an ordinary
// IEEE fma, so a row's bits never depend on which pass or pairing it had.
//
// Data movement: the RB activation rows live in shared memory, split into
// low/high float4 halves so a warp's reads are conflict-free; each warp
// streams NV = 8 consecutive vocab rows at a time with 16-byte
// non-allocating loads (one 512-byte coalesced segment per row per step),
// prefetching the next step while the current one is multiplied.  With more
// than RB rows the weights are streamed once per pass of RB rows.
#include <algorithm>

#include "vr_common.cuh"
#include "vr_kernels.h"

namespace vr {
namespace ffma {

constexpr int NV = 8;               // vocab rows per warp task
constexpr int WARPS = 8;
constexpr int THREADS = WARPS * 32;
constexpr int MAX_SMEM = 200 * 1024;

// Weights are read once per call: no L1 allocation, and evict-first in L2 so
// that the stream does not push the logits, activations or the next
// kernels' code out of L2.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p, uint64_t policy) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(policy));
  return v;
}

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

template <int RB>
__global__ void __launch_bounds__(THREADS, 1)
    project_ffma_kernel(const uint16_t* __restrict__ weight, const float* __restrict__ act,
                        int hidden, int vocab, int row_base, float* __restrict__ logits) {
  extern __shared__ float4 sA[];               // [2][RB][chunks]
  pdl_trigger();
  pdl_wait();
  const int chunks = hidden / 8;
  float4* sLo = sA;
  float4* sHi = sA + RB * chunks;
  for (int i = threadIdx.x; i < RB * chunks; i += THREADS) {
    const int r = i / chunks, c = i % chunks;
    const float* a = act + static_cast<size_t>(row_base + r) * hidden + c * 8;
    sLo[i] = make_float4(a[0], a[1], a[2], a[3]);
    sHi[i] = make_float4(a[4], a[5], a[6], a[7]);
  }
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int steps = (chunks + 31) / 32;
  const uint64_t pol = l2_policy_evict_first();
  const long long n_tasks = (static_cast<long long>(vocab) + NV - 1) / NV;
  const long long gw = static_cast<long long>(blockIdx.x) * WARPS + warp;
  const long long tw = static_cast<long long>(gridDim.x) * WARPS;
  const long long t_begin = gw * n_tasks / tw, t_end = (gw + 1) * n_tasks / tw;

  for (long long task = t_begin; task < t_end; ++task) {
    const long long v0 = task * NV;
    const uint4* wrow[NV];
#pragma unroll
    for (int n = 0; n < NV; ++n) {
      const long long v = min(v0 + n, static_cast<long long>(vocab) - 1);
      wrow[n] = reinterpret_cast<const uint4*>(weight + v * hidden);
    }
    float2 acc[NV / 2][RB];
#pragma unroll
    for (int p = 0; p < NV / 2; ++p)
#pragma unroll
      for (int r = 0; r < RB; ++r) acc[p][r] = make_float2(0.f, 0.f);

    uint4 cur[NV];
    {
      const int c = lane;
#pragma unroll
      for (int n = 0; n < NV; ++n) cur[n] = (c < chunks) ? ld_stream(wrow[n] + c, pol) : make_uint4(0, 0, 0, 0);
    }
    for (int j = 0; j < steps; ++j) {
      const int c = lane + 32 * j;
      const int cn = c + 32;
      uint4 nxt[NV];
#pragma unroll
      for (int n = 0; n < NV; ++n)
        nxt[n] = (j + 1 < steps && cn < chunks) ? ld_stream(wrow[n] + cn, pol) : make_uint4(0, 0, 0, 0);
      if (c < chunks) {
#pragma unroll
        for (int r = 0; r < RB; ++r) {
          const float4 lo = sLo[r * chunks + c];
          const float4 hi = sHi[r * chunks + c];
          const float a[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
          for (int p = 0; p < NV / 2; ++p) {
            const uint32_t* u0 = reinterpret_cast<const uint32_t*>(&cur[2 * p]);
            const uint32_t* u1 = reinterpret_cast<const uint32_t*>(&cur[2 * p + 1]);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              acc[p][r] = __ffma2_rn(make_float2(bf_lo(u0[q]), bf_lo(u1[q])),
                                     make_float2(a[2 * q], a[2 * q]), acc[p][r]);
              acc[p][r] = __ffma2_rn(make_float2(bf_hi(u0[q]), bf_hi(u1[q])),
                                     make_float2(a[2 * q + 1], a[2 * q + 1]), acc[p][r]);
            }
          }
        }
      }
#pragma unroll
      for (int n = 0; n < NV; ++n) cur[n] = nxt[n];
    }
    // xor-butterfly across the 32 lanes, fixed order
#pragma unroll
    for (int p = 0; p < NV / 2; ++p)
#pragma unroll
      for (int r = 0; r < RB; ++r) {
        float x = acc[p][r].x, y = acc[p][r].y;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
          x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, o));
          y = __fadd_rn(y, __shfl_xor_sync(0xffffffffu, y, o));
        }
        acc[p][r] = make_float2(x, y);
      }
    // lane (n * RB + r) % 32 stores output (r, v0 + n)
#pragma unroll
    for (int p = 0; p < NV / 2; ++p)
#pragma unroll
      for (int r = 0; r < RB; ++r)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int n = 2 * p + h;
          if (lane == ((n * RB + r) & 31) && v0 + n < vocab)
            logits[static_cast<size_t>(row_base + r) * vocab + v0 + n] = h ? acc[p][r].y : acc[p][r].x;
        }
  }
}

template <int RB>
int launch_pass(const uint16_t* weight, const float* act, int hidden, int vocab, int row_base,
                float* logits, int sms, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(2) * RB * (hidden / 8) * sizeof(float4);
  if (cudaFuncSetAttribute(project_ffma_kernel<RB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return VR_ERR_CUDA;
  return launch_pdl(project_ffma_kernel<RB>, dim3(sms), dim3(THREADS), smem, stream, weight, act,
                    hidden, vocab, row_base, logits) == cudaSuccess
             ? VR_OK
             : VR_ERR_CUDA;
}

}  // namespace ffma

int ffma_rows_per_pass(int hidden) {
  const int per_row = 2 * (hidden / 8) * static_cast<int>(sizeof(float4));
  return std::min(8, ffma::MAX_SMEM / per_row);
}

int launch_project_ffma(const uint16_t* weight, const float* act, int rows, int hidden, int vocab,
                        float* logits, cudaStream_t stream) {
  const int rb_max = ffma_rows_per_pass(hidden);
  if (rb_max < 1) return VR_ERR_UNSUPPORTED;
  const int sms = device_sm_count();
  if (sms <= 0) return VR_ERR_CUDA;
  for (int r0 = 0; r0 < rows; r0 += rb_max) {
    const int rb = std::min(rb_max, rows - r0);
    int st;
    switch (rb) {
      case 1: st = ffma::launch_pass<1>(weight, act, hidden, vocab, r0, logits, sms, stream); break;
      case 2: st = ffma::launch_pass<2>(weight, act, hidden, vocab, r0, logits, sms, stream); break;
      case 3: st = ffma::launch_pass<3>(weight, act, hidden, vocab, r0, logits, sms, stream); break;
      case 4: st = ffma::launch_pass<4>(weight, act, hidden, vocab, r0, logits, sms, stream); break;
      case 5: st = ffma::launch_pass<5>(weight, act, hidden, vocab, r0, logits, sms, stream); break;
      case 6: st = ffma::launch_pass<6>(weight, act, hidden, vocab, r0, logits, sms, stream); break;
      case 7: st = ffma::launch_pass<7>(weight, act, hidden, vocab, r0, logits, sms, stream); break;
      default: st = ffma::launch_pass<8>(weight, act, hidden, vocab, r0, logits, sms, stream); break;
    }
    if (st != VR_OK) return st;
  }
  return VR_OK;
}

}  // namespace vr
