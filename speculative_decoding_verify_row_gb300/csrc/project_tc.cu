// Verify projection on the 5th-generation tensor cores (tcgen05).
//
//   logits[r][v] = sum_h W[v][h] * A[r][h]      (W bf16 [V][H], A fp32 [R][H])
//
// "Speculative decoding on RDNA" §01: the weights are read once for all
// verify rows; §02: a row's sum must not depend on how many rows share the
// pass.  Design for sm_103a:
//
//  * The fp32 activations are split exactly into three bf16 planes
//    (a = hi + mid + lo; 8 + 8 + 8 significand bits cover float32's 24), so
//    every product W*plane is exact and the tensor core adds exact
//    products in fp32.  The planes of 32 rows are stacked as the N = 96
//    columns of one MMA; the epilogue adds (hi + mid) + lo.
//  * Every launch uses the same instruction shape (M = 128 vocab rows,
//    N = 96, K = 16) and the same K order whatever the row count: rows past
//    R are zero columns.  Row r's bits therefore do not depend on R.
//  * Each CTA (one per SM, persistent) walks units of two 128-row vocab
//    tiles.  Warp 0 streams W tiles (2 x 16 KB) and the shared plane tile
//    (12 KB) per 64-wide K block through a 5-stage TMA ring; one thread of
//    warp 1 issues the MMAs into a double-buffered TMEM accumulator
//    (2 x 192 columns); warps 2-5 drain TMEM and write the logits, so the
//    epilogue of one unit overlaps the weight stream of the next.
//  * Optionally the epilogue also records, per row and per 32 vocabulary
//    rows, the largest order key (a warp max), which lets the sampling stage
//    find a row's top 64 without reading the whole row.
//  * All mbarrier waits are bounded: on time-out the CTA records
//    VR_DEV_TIMEOUT, drains what it issued, frees TMEM and returns.
#include <algorithm>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "tc_common.cuh"
#include "vr_common.cuh"
#include "vr_kernels.h"

namespace vr {
namespace tc {

constexpr int BM = 128;                  // vocab rows per tile (MMA M)
constexpr int BK = 64;                   // hidden per K block (128 B of bf16)
constexpr int NP = 32;                   // verify rows per plane group
constexpr int NPLANE = 3;
constexpr int BN = NP * NPLANE;          // 96 MMA columns
constexpr int MT = 2;                    // vocab tiles per unit
constexpr int STAGES = 5;
constexpr int W_TILE_BYTES = BM * BK * 2;            // 16384
constexpr int B_TILE_BYTES = BN * BK * 2;            // 12288
constexpr int STAGE_BYTES = MT * W_TILE_BYTES + B_TILE_BYTES;
constexpr int TMEM_COLS_PER_BUF = MT * BN;           // 192
constexpr int TMEM_ALLOC = 512;
constexpr int THREADS = 192;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// instruction descriptor, kind::f16: D f32 (bits 4-5 = 1), A bf16 (7-9 = 1),
// B bf16 (10-12 = 1), both K-major, N >> 3 at bits 17-22, M >> 4 at 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                            ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

using namespace tcx;

__global__ void __launch_bounds__(THREADS, 1)
    project_tc_kernel(const __grid_constant__ CUtensorMap tm_w,
                      const __grid_constant__ CUtensorMap tm_b, int hidden, int vocab,
                      int rows_in_group, int row_base, float* __restrict__ logits,
                      uint32_t* __restrict__ gmax, int ngroups, int32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  // barrier slots: full[STAGES], empty[STAGES], tmem_full[2], tmem_empty[2]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_mtiles = (vocab + BM - 1) / BM;
  const int n_units = (n_mtiles + MT - 1) / MT;
  const int n_kb = (hidden + BK - 1) / BK;

  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + STAGES + s); };
  auto tfull_bar = [&](int b) { return smem_u32(bars + 2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return smem_u32(bars + 2 * STAGES + 2 + b); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 4 * 32);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_w)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_b)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_holder)),
                 "r"(TMEM_ALLOC)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // the prologue above overlaps the previous kernel; from here on the planes
  // and the logits buffer are touched, so wait for it to complete
  pdl_trigger();
  pdl_wait();

  if (warp == 0) {
    // ---------------- producer: TMA ring ----------------
    if (lane == 0) {
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_b = l2_policy_evict_last();
      int s = 0;
      uint32_t ph = 0;
      int last_fill_parity[STAGES];
      for (int i = 0; i < STAGES; ++i) last_fill_parity[i] = -1;
      for (int u = blockIdx.x; u < n_units && !*abort_flag; u += gridDim.x) {
        const int nmt = min(MT, n_mtiles - u * MT);
        const uint32_t bytes = nmt * W_TILE_BYTES + B_TILE_BYTES;
        for (int kb = 0; kb < n_kb; ++kb) {
          if (!mbar_wait(empty_bar(s), ph ^ 1, abort_flag, status)) break;
          mbar_expect_tx(full_bar(s), bytes);
          uint8_t* st = smem + s * STAGE_BYTES;
          for (int mt = 0; mt < nmt; ++mt)
            tma_load_2d(smem_u32(st + mt * W_TILE_BYTES), &tm_w, kb * BK, (u * MT + mt) * BM,
                        full_bar(s), pol_w);
          tma_load_2d(smem_u32(st + MT * W_TILE_BYTES), &tm_b, kb * BK, 0, full_bar(s), pol_b);
          last_fill_parity[s] = static_cast<int>(ph);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1;
          }
        }
      }
      if (*abort_flag) {
        // drain: wait (bounded) until the last fill of every stage has landed,
        // so that no bulk copy is still writing when the CTA exits
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
      int buf = 0;
      uint32_t bph = 0;
      const uint32_t a0 = smem_u32(smem);
      for (int u = blockIdx.x; u < n_units && !*abort_flag; u += gridDim.x) {
        const int nmt = min(MT, n_mtiles - u * MT);
        if (!mbar_wait(tempty_bar(buf), bph ^ 1, abort_flag, status)) break;
        tc_fence_after();
        const uint32_t dcol = tmem_base + buf * TMEM_COLS_PER_BUF;
        bool ok = true;
        for (int kb = 0; kb < n_kb; ++kb) {
          if (!mbar_wait(full_bar(s), ph, abort_flag, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = a0 + s * STAGE_BYTES;
          const uint64_t bdesc = sw128_desc(st + MT * W_TILE_BYTES);
          for (int mt = 0; mt < nmt; ++mt) {
            const uint64_t adesc = sw128_desc(st + mt * W_TILE_BYTES);
#pragma unroll
            for (int ks = 0; ks < BK / 16; ++ks) {
              // advance 16 bf16 = 32 bytes along K inside the swizzled row
              mma_bf16_desc(dcol + mt * BN, adesc + 2 * ks, bdesc + 2 * ks, kIdesc,
                            (kb | ks) ? 1u : 0u);
            }
          }
          mma_commit(empty_bar(s));
          if (++s == STAGES) {
            s = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        mma_commit(tfull_bar(buf));
        buf ^= 1;
        if (buf == 0) bph ^= 1;
      }
      if (*abort_flag) {
        // make sure every MMA issued so far has finished before TMEM is freed
        mma_commit(tfull_bar(buf));
        const long long t0 = clock64();
        while (!mbar_try_wait(tfull_bar(buf), bph) && clock64() - t0 < kWaitLimitCycles / 8) {
        }
      }
    }
  } else {
    // ---------------- epilogue: TMEM -> registers -> logits ----------------
    const int quarter = warp & 3;                 // TMEM lanes this warp may read
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    int buf = 0;
    uint32_t bph = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      const int nmt = min(MT, n_mtiles - u * MT);
      const bool ok = mbar_wait(tfull_bar(buf), bph, abort_flag, status);
      __syncwarp();
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint32_t dcol = tmem_base + lane_off + buf * TMEM_COLS_PER_BUF;
      for (int mt = 0; mt < nmt; ++mt) {
        const int vbase = (u * MT + mt) * BM + quarter * 32;     // this warp's 32 vocab rows
        const int v = vbase + lane;
        for (int rb = 0; rb < rows_in_group; rb += 8) {
          float hi[8], mid[8], lo[8];
          tmem_ld8(dcol + mt * BN + 0 * NP + rb, hi);
          tmem_ld8(dcol + mt * BN + 1 * NP + rb, mid);
          tmem_ld8(dcol + mt * BN + 2 * NP + rb, lo);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int r = rb + i;
            if (r < rows_in_group) {
              const float x = __fadd_rn(__fadd_rn(hi[i], mid[i]), lo[i]);
              if (v < vocab) logits[static_cast<size_t>(row_base + r) * vocab + v] = x;
              if (gmax && vbase < vocab) {
                // the largest order key of these 32 vocabulary rows
                const uint32_t k =
                    __reduce_max_sync(0xffffffffu, v < vocab ? float_key(x) : 0u);
                if (lane == 0) gmax[static_cast<size_t>(row_base + r) * ngroups + (vbase >> 5)] = k;
              }
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(tempty_bar(buf));
      buf ^= 1;
      if (buf == 0) bph ^= 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_ALLOC)
                 : "memory");
  }
}

// A [R][H] fp32 -> planes [G][96][H] bf16: plane p of row r of group g sits
// at plane-row p * 32 + (r - 32 g); rows past R are zero.  hi = RN(a),
// mid = RN(a - hi), lo = RN(a - hi - mid); both subtractions are exact.
__global__ void split_planes_kernel(const float* __restrict__ act, int rows, int hidden,
                                    int groups, __nv_bfloat16* __restrict__ planes) {
  pdl_trigger();
  pdl_wait();
  const int chunks = hidden / 8;
  const long long total = static_cast<long long>(groups) * NP * chunks;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(i % chunks);
    const int rr = static_cast<int>(i / chunks);       // g * 32 + local row
    const int g = rr / NP, rl = rr % NP;
    const int r = rr;                                  // global row
    __align__(16) __nv_bfloat16 h[8], m[8], l[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float a = (r < rows) ? act[static_cast<size_t>(r) * hidden + c * 8 + j] : 0.f;
      const __nv_bfloat16 bh = __float2bfloat16_rn(a);
      const float r1 = __fsub_rn(a, __bfloat162float(bh));
      const __nv_bfloat16 bm = __float2bfloat16_rn(r1);
      const float r2 = __fsub_rn(r1, __bfloat162float(bm));
      h[j] = bh;
      m[j] = bm;
      l[j] = __float2bfloat16_rn(r2);
    }
    const size_t base = (static_cast<size_t>(g) * BN + rl) * hidden + c * 8;
    *reinterpret_cast<uint4*>(planes + base) = *reinterpret_cast<const uint4*>(h);
    *reinterpret_cast<uint4*>(planes + base + static_cast<size_t>(NP) * hidden) =
        *reinterpret_cast<const uint4*>(m);
    *reinterpret_cast<uint4*>(planes + base + static_cast<size_t>(2 * NP) * hidden) =
        *reinterpret_cast<const uint4*>(l);
  }
}

}  // namespace tc

// ---------------------------------------------------------------------------
// host side

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool get_encoder() {
  if (g_encode) return true;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return false;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return true;
}

int g_num_sms = 0;
bool g_attr_set = false;
}  // namespace

// 2-D bf16 tensor map over a row-major [outer][inner] array, tiles of
// box_outer x box_inner elements, 128-byte swizzle (box_inner * 2 == 128).
bool encode_bf16_tile(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                      uint32_t box_inner, uint32_t box_outer) {
  if (!get_encoder()) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t tc_plane_bytes(int rows, int hidden) {
  const int groups = (rows + tc::NP - 1) / tc::NP;
  return static_cast<size_t>(groups) * tc::BN * hidden * 2;
}

int launch_project_tc(const uint16_t* weight, const float* act, int rows, int hidden, int vocab,
                      float* logits, void* planes, uint32_t* gmax, int32_t* status,
                      cudaStream_t stream) {
  if (!g_num_sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return VR_ERR_CUDA;
    if (cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return VR_ERR_CUDA;
  }
  if (!g_attr_set) {
    if (cudaFuncSetAttribute(tc::project_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             tc::SMEM_BYTES) != cudaSuccess)
      return VR_ERR_CUDA;
    g_attr_set = true;
  }
  const int groups = (rows + tc::NP - 1) / tc::NP;
  auto* pl = static_cast<__nv_bfloat16*>(planes);
  {
    const long long work = static_cast<long long>(groups) * tc::NP * (hidden / 8);
    const int threads = 256;
    const int blocks = static_cast<int>(std::min<long long>((work + threads - 1) / threads,
                                                            static_cast<long long>(g_num_sms) * 8));
    if (launch_pdl(tc::split_planes_kernel, dim3(blocks), dim3(threads), 0, stream, act, rows,
                   hidden, groups, pl) != cudaSuccess)
      return VR_ERR_CUDA;
  }
  CUtensorMap tm_w;
  if (!encode_bf16_tile(&tm_w, weight, hidden, vocab, tc::BK, tc::BM)) return VR_ERR_ARG;
  const int n_mtiles = (vocab + tc::BM - 1) / tc::BM;
  const int n_units = (n_mtiles + tc::MT - 1) / tc::MT;
  const int grid = std::min(n_units, g_num_sms);
  for (int g = 0; g < groups; ++g) {
    CUtensorMap tm_b;
    if (!encode_bf16_tile(&tm_b, pl + static_cast<size_t>(g) * tc::BN * hidden, hidden, tc::BN,
                          tc::BK, tc::BN))
      return VR_ERR_ARG;
    const int rg = std::min(tc::NP, rows - g * tc::NP);
    if (launch_pdl(tc::project_tc_kernel, dim3(grid), dim3(tc::THREADS), tc::SMEM_BYTES, stream,
                   tm_w, tm_b, hidden, vocab, rg, g * tc::NP, logits, gmax,
                   (vocab + 31) / 32, status) != cudaSuccess)
      return VR_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? VR_OK : VR_ERR_CUDA;
}

}  // namespace vr
