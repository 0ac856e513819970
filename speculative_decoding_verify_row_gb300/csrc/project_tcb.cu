// Verify projection for many verify rows at once (batched serving) on the
// 5th-generation tensor cores.
//
//   logits[r][v] = sum_h W[v][h] * A[r][h]      (W bf16 [V][H], A fp32 [R][H])
//
// With hundreds of rows ("a request table of many requests") the product is
// a dense contraction and the tensor pipe, not HBM, sets the pace.  Design:
//
//  * Roles: the activation rows are the MMA's M operand (two 128-row halves,
//    256 rows per group) and a 256-row tile of the vocabulary is N.  Each
//    CTA keeps two TMEM accumulators of 128 lanes x 256 columns (all 512
//    columns) and streams its vocabulary tiles' weights once per group.
//  * Precision: each fp32 activation is split exactly into two bf16 planes,
//    hi = RN(a) and lo = RN(a - hi), which keep 16 significant bits (error
//    below 2^-17 |a|).  Products with the bf16 weights are exact and both
//    planes accumulate into the same fp32 accumulator, plane hi then plane
//    lo for every 64-wide K block.
//  * Row-count invariance: every group is one 256-row MMA shape with zero
//    rows past R, and the K order is fixed, so a row's bits do not depend
//    on how many rows share the call (within this path).
//  * Warp 0 feeds a 2-stage TMA ring (32 KB of weights, evict-first in L2,
//    and 64 KB of plane tiles, evict-last, per stage), one thread of warp 1
//    issues M128 N256 K16 MMAs, warps 2-5 drain TMEM into the logits.  The
//    accumulator fills all of TMEM, so the next tile's MMAs wait for the
//    drain: the drain therefore only moves TMEM through two 16 KB staging
//    buffers in shared memory (128-byte swizzled rows) and tensor stores
//    write the logits to global memory in the background.
//  * Optionally the epilogue records, per row and per 32 vocabulary rows, the
//    largest order key (the sampling stage's filter).
//  * All waits are bounded (VR_DEV_TIMEOUT), as in the chain projection.
#include <algorithm>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "tc_common.cuh"
#include "vr_common.cuh"
#include "vr_kernels.h"

namespace vr {
namespace tcb {

using namespace tcx;

constexpr int BM = 128;                      // activation rows per MMA (M)
constexpr int MH = 2;                        // M halves
constexpr int GROUP = BM * MH;               // 256 rows per group
constexpr int BN = 256;                      // vocabulary rows per tile (N)
constexpr int BK = 64;
constexpr int NPLANE = 2;
constexpr int STAGES = 2;
constexpr int W_TILE_BYTES = BN * BK * 2;                                  // 32768
constexpr int A_TILE_BYTES = BM * BK * 2;                                  // 16384
constexpr int STAGE_BYTES = W_TILE_BYTES + NPLANE * MH * A_TILE_BYTES;     // 98304
constexpr int TMEM_COLS = MH * BN;                                         // 512
constexpr int THREADS = 192;
constexpr int OUT_COLS = 32;                                               // per staged box
constexpr int OUT_BYTES = BM * OUT_COLS * 4;                               // 16384
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 2 * OUT_BYTES + 1024 + 256;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// kind::f16 instruction descriptor: D f32, A and B bf16, both K-major,
// N = 256, M = 128
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                            ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

__global__ void __launch_bounds__(THREADS, 1)
    project_tcb_kernel(const __grid_constant__ CUtensorMap tm_w,
                       const __grid_constant__ CUtensorMap tm_a,
                       const __grid_constant__ CUtensorMap tm_out,
                       const __grid_constant__ CUtensorMap tm_out2, int staged, int hidden,
                       int vocab, int rows_in_group, int row_base, float* __restrict__ logits,
                       float* __restrict__ logits2, int vec_ok, uint32_t* __restrict__ gmax,
                       int ngroups, int32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* out_stage = smem + STAGES * STAGE_BYTES;               // 2 x 16 KB, 1024-aligned
  uint64_t* bars = reinterpret_cast<uint64_t*>(out_stage + 2 * OUT_BYTES);
  // barrier slots: full[STAGES], empty[STAGES], tmem_full, tmem_empty
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_tiles = (vocab + BN - 1) / BN;
  const int n_kb = (hidden + BK - 1) / BK;

  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + STAGES + s); };
  const uint32_t tfull = smem_u32(bars + 2 * STAGES);
  const uint32_t tempty = smem_u32(bars + 2 * STAGES + 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, 4 * 32);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_w)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_a)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_holder)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncwarp();     // lanes of warps 0 and 1 took single-lane branches above
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  pdl_wait();
  // a window starts with this kernel: its dependents may launch only now,
  // once every kernel before the window is complete, because the later
  // kernels of the window read the window's inputs before their own wait
  pdl_trigger();

  if (warp == 0) {
    // ---------------- producer ----------------
    if (lane == 0) {
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_a = l2_policy_evict_last();
      int s = 0;
      uint32_t ph = 0;
      int last_fill_parity[STAGES];
      for (int i = 0; i < STAGES; ++i) last_fill_parity[i] = -1;
      for (int t = blockIdx.x; t < n_tiles && !*abort_flag; t += gridDim.x) {
        for (int kb = 0; kb < n_kb; ++kb) {
          if (!mbar_wait(empty_bar(s), ph ^ 1, abort_flag, status)) break;
          mbar_expect_tx(full_bar(s), STAGE_BYTES);
          uint8_t* st = smem + s * STAGE_BYTES;
          tma_load_2d(smem_u32(st), &tm_w, kb * BK, t * BN, full_bar(s), pol_w);
          for (int p = 0; p < NPLANE; ++p)
            for (int mh = 0; mh < MH; ++mh)
              tma_load_2d(smem_u32(st + W_TILE_BYTES + (p * MH + mh) * A_TILE_BYTES), &tm_a,
                          kb * BK, p * GROUP + mh * BM, full_bar(s), pol_a);
          last_fill_parity[s] = static_cast<int>(ph);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1;
          }
        }
      }
      if (*abort_flag) {
        for (int i = 0; i < STAGES; ++i) {
          if (last_fill_parity[i] < 0) continue;
          const long long t0 = clock64();
          while (!mbar_try_wait(full_bar(i), static_cast<uint32_t>(last_fill_parity[i])) &&
                 clock64() - t0 < kWaitLimitCycles / 8) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      uint32_t tph = 0;
      const uint32_t a0 = smem_u32(smem);
      for (int t = blockIdx.x; t < n_tiles && !*abort_flag; t += gridDim.x) {
        if (!mbar_wait(tempty, tph ^ 1, abort_flag, status)) break;
        tc_fence_after();
        bool ok = true;
        for (int kb = 0; kb < n_kb; ++kb) {
          if (!mbar_wait(full_bar(s), ph, abort_flag, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = a0 + s * STAGE_BYTES;
          const uint64_t bdesc = sw128_desc(st);
          for (int mh = 0; mh < MH; ++mh)
            for (int p = 0; p < NPLANE; ++p) {
              const uint64_t adesc = sw128_desc(st + W_TILE_BYTES + (p * MH + mh) * A_TILE_BYTES);
#pragma unroll
              for (int ks = 0; ks < BK / 16; ++ks)
                mma_bf16_desc(tmem_base + mh * BN, adesc + 2 * ks, bdesc + 2 * ks, kIdesc,
                              (kb | p | ks) ? 1u : 0u);
            }
          mma_commit(empty_bar(s));
          if (++s == STAGES) {
            s = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        mma_commit(tfull);
        tph ^= 1;
      }
      if (*abort_flag) {
        mma_commit(tfull);
        const long long t0 = clock64();
        while (!mbar_try_wait(tfull, tph) && clock64() - t0 < kWaitLimitCycles / 8) {
        }
      }
    }
  } else {
    // ---------------- epilogue ----------------
    const int quarter = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const bool vec = vec_ok != 0;           // 16-byte aligned rows: float4 stores
    const int et = threadIdx.x - 64;        // epilogue thread 0..127
    int box = 0;                            // staged boxes issued so far
    uint32_t tph = 0;
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x) {
      const bool okw = mbar_wait(tfull, tph, abort_flag, status);
      __syncwarp();
      if (!__all_sync(0xffffffffu, okw)) break;
      tc_fence_after();
      for (int mh = 0; mh < MH; ++mh) {
        const int rl = mh * BM + quarter * 32 + lane;           // row within the group
        float* out = logits + static_cast<size_t>(row_base + rl) * vocab;
        // a second copy of the row (penalised in place later), or none
        float* out2 = logits2 ? logits2 + static_cast<size_t>(row_base + rl) * vocab : nullptr;
        for (int c = 0; c < BN / 32; ++c) {
          float v[32];
          tmem_ld32(tmem_base + lane_off + mh * BN + c * 32, v);
          tmem_ld_wait();
          const int v0 = t * BN + c * 32;
          if (gmax && rl < rows_in_group && v0 < vocab) {
            // the largest order key of these 32 vocabulary rows of this row
            uint32_t k = 0u;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const uint32_t ki = (v0 + i < vocab) ? float_key(v[i]) : 0u;
              k = ki > k ? ki : k;
            }
            gmax[static_cast<size_t>(row_base + rl) * ngroups + (v0 >> 5)] = k;
          }
          if (staged) {
            // row rl's 32 values into the staging box (row quarter*32 + lane,
            // 16-byte chunk k at position k ^ (row & 7)), then one tensor
            // store per output; the buffer is reused two boxes later, after
            // the store that read it
            const int b = box & 1;
            uint8_t* buf = out_stage + b * OUT_BYTES;
            if (et == 0) bulk_wait_read<1>();
            named_sync(1, 128);
            const int srow = quarter * 32 + lane;
#pragma unroll
            for (int k = 0; k < 8; ++k)
              *reinterpret_cast<float4*>(buf + srow * 128 + ((k ^ (srow & 7)) << 4)) =
                  make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            named_sync(1, 128);
            if (et == 0) {
              tma_store_2d(&tm_out, smem_u32(buf), v0, row_base + mh * BM);
              if (logits2) tma_store_2d(&tm_out2, smem_u32(buf), v0, row_base + mh * BM);
              bulk_commit();
            }
            ++box;
          } else if (rl < rows_in_group) {
            if (vec && v0 + 32 <= vocab) {
#pragma unroll
              for (int i = 0; i < 8; ++i)
                *reinterpret_cast<float4*>(out + v0 + 4 * i) =
                    make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
              if (out2)
#pragma unroll
                for (int i = 0; i < 8; ++i)
                  *reinterpret_cast<float4*>(out2 + v0 + 4 * i) =
                      make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
            } else {
              for (int i = 0; i < 32; ++i)
                if (v0 + i < vocab) out[v0 + i] = v[i];
              if (out2)
                for (int i = 0; i < 32; ++i)
                  if (v0 + i < vocab) out2[v0 + i] = v[i];
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(tempty);
      tph ^= 1;
    }
  }

  // the tensor stores issued by the epilogue have written their data
  if (staged && threadIdx.x == 64) bulk_wait_all();
  tc_fence_before();
  // Each role above runs on one lane of its warp (producer, MMA issuer) while
  // the other lanes come straight here, so a warp's lanes reach this point at
  // different times.  The block barrier counts arrivals per warp, so a warp
  // must arrive as a whole: without the reconvergence below, the same barrier
  // of the chain projection kernel was measured to release while its
  // epilogue warps were still reading TMEM, and the dealloc that follows it
  // could then free TMEM in use.
  __syncwarp();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

// A [R][H] fp32 -> planes [G][2][256][H] bf16: hi = RN(a), lo = RN(a - hi)
// (the subtraction is exact); rows past R are zero.
__global__ void split_planes2_kernel(const float* __restrict__ act, int rows, int hidden,
                                     int groups, __nv_bfloat16* __restrict__ planes) {
  // the projection that follows reads only the weights before its own
  // wait, so it may launch at once and start its weight stream; the kernels
  // after it launch only once it is past its wait
  pdl_trigger();
  pdl_wait();
  const int chunks = hidden / 8;
  const long long total = static_cast<long long>(groups) * GROUP * chunks;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(i % chunks);
    const int r = static_cast<int>(i / chunks);           // global row
    const int g = r / GROUP, rl = r % GROUP;
    __align__(16) __nv_bfloat16 h[8], l[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float a = (r < rows) ? act[static_cast<size_t>(r) * hidden + c * 8 + j] : 0.f;
      const __nv_bfloat16 bh = __float2bfloat16_rn(a);
      h[j] = bh;
      l[j] = __float2bfloat16_rn(__fsub_rn(a, __bfloat162float(bh)));
    }
    const size_t base = (static_cast<size_t>(g) * NPLANE * GROUP + rl) * hidden + c * 8;
    *reinterpret_cast<uint4*>(planes + base) = *reinterpret_cast<const uint4*>(h);
    *reinterpret_cast<uint4*>(planes + base + static_cast<size_t>(GROUP) * hidden) =
        *reinterpret_cast<const uint4*>(l);
  }
}

}  // namespace tcb

namespace {
}  // namespace

size_t tcb_plane_bytes(int rows, int hidden) {
  const int groups = (rows + tcb::GROUP - 1) / tcb::GROUP;
  return static_cast<size_t>(groups) * tcb::NPLANE * tcb::GROUP * hidden * 2;
}

int launch_project_tcb(const uint16_t* weight, const float* act, int rows, int hidden, int vocab,
                       float* logits, float* logits2, void* planes, uint32_t* gmax,
                       int32_t* status, cudaStream_t stream) {
  const int num_sms = device_sm_count();
  if (num_sms <= 0) return VR_ERR_CUDA;
  static std::atomic<bool> attr_set[kMaxDevices];
  if (set_smem_limit_once(tcb::project_tcb_kernel, tcb::SMEM_BYTES, attr_set) != cudaSuccess)
    return VR_ERR_CUDA;
  const int groups = (rows + tcb::GROUP - 1) / tcb::GROUP;
  auto* pl = static_cast<__nv_bfloat16*>(planes);
  {
    const long long work = static_cast<long long>(groups) * tcb::GROUP * (hidden / 8);
    const int threads = 256;
    const int blocks = static_cast<int>(std::min<long long>((work + threads - 1) / threads,
                                                            static_cast<long long>(num_sms) * 8));
    if (launch_pdl(tcb::split_planes2_kernel, dim3(blocks), dim3(threads), 0, stream, act, rows,
                   hidden, groups, pl) != cudaSuccess)
      return VR_ERR_CUDA;
  }
  CUtensorMap tm_w;
  if (!encode_bf16_tile(&tm_w, weight, hidden, vocab, tcb::BK, tcb::BN)) return VR_ERR_ARG;
  const int n_tiles = (vocab + tcb::BN - 1) / tcb::BN;
  const int grid = std::min(n_tiles, num_sms);
  const int vec_ok = (vocab % 4 == 0) && (reinterpret_cast<uintptr_t>(logits) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(logits2) % 16 == 0);
  // the staged epilogue's tensor stores: fp32 boxes of 32 columns x 128 rows
  // (row stride vocab * 4 must be a multiple of 16 bytes, bases 16-aligned)
  CUtensorMap tm_out{}, tm_out2{};
  int staged = vec_ok && encode_f32_box_sw128(&tm_out, logits, vocab, rows, tcb::OUT_COLS, tcb::BM);
  if (staged && logits2)
    staged = encode_f32_box_sw128(&tm_out2, logits2, vocab, rows, tcb::OUT_COLS, tcb::BM);
  for (int g = 0; g < groups; ++g) {
    CUtensorMap tm_a;
    if (!encode_bf16_tile(&tm_a, pl + static_cast<size_t>(g) * tcb::NPLANE * tcb::GROUP * hidden,
                          hidden, tcb::NPLANE * tcb::GROUP, tcb::BK, tcb::BM))
      return VR_ERR_ARG;
    const int rg = std::min(tcb::GROUP, rows - g * tcb::GROUP);
    if (launch_pdl(tcb::project_tcb_kernel, dim3(grid), dim3(tcb::THREADS), tcb::SMEM_BYTES,
                   stream, tm_w, tm_a, tm_out, tm_out2, staged, hidden, vocab, rg,
                   g * tcb::GROUP, logits, logits2, vec_ok, gmax, (vocab + 31) / 32,
                   status) != cudaSuccess)
      return VR_ERR_CUDA;
  }
  return VR_OK;
}

}  // namespace vr
