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
//    tiles.  Per 64-wide K block, one thread of warp 0 streams the unit's
//    256 x 64 W block (32 KB) through a 5-stage TMA ring together with the
//    block's plane tile (96 x 64 bf16, in the 128-byte swizzled layout the
//    MMA reads).  The W block is one 256-row box: the same bytes and
//    shared-memory layout as two 128-row boxes with one TMA instruction
//    (a TMA-only stream of these weights ran faster with the single box).
//    In the last unit of an odd tile count its second half lies past the
//    vocabulary and is zero-filled by the TMA; no MMA reads it.  For up to 16 rows the planes are built in the kernel: the TMA
//    brings the group's fp32 activations for the block (R x 64) into the
//    end of the plane tile and warp 6 splits them in place, so no separate
//    pass runs before the projection.  For more rows one warp cannot keep
//    pace with the weight stream, so a split kernel writes the planes of
//    every group first and the TMA loads plane tiles.  One thread of warp 1
//    issues the MMAs into a double-buffered TMEM accumulator (2 x 192
//    columns); warps 2-5 drain TMEM and write the logits, so the epilogue of
//    one unit overlaps the weight stream of the next.
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
constexpr int THREADS = 224;              // 7 warps: TMA, MMA, 4 x epilogue, planes
constexpr int PLANE_WARP = 6;
constexpr int FUSED_MAX_ROWS = 16;        // planes built in the kernel up to this many rows
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// instruction descriptor, kind::f16: D f32 (bits 4-5 = 1), A bf16 (7-9 = 1),
// B bf16 (10-12 = 1), both K-major, N >> 3 at bits 17-22, M >> 4 at 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                            ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

using namespace tcx;

// (lo, hi) rounded to bf16 (nearest, ties to even) and packed, lo in the low
// half: one conversion instruction for two values.
__device__ __forceinline__ uint32_t bf16x2_rn(float2 x) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(x.x, x.y);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// the two bf16 of a packed pair as floats (exact)
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t p) {
  return make_float2(__uint_as_float(p << 16), __uint_as_float(p & 0xffff0000u));
}

// Plane tiles, built in the kernel (groups of at most 16 rows).  The TMA
// lands the group's activations for one K block, act[row_base + r][kb*64 ..
// + 64) for r < R (zeros past hidden), as R rows of 256 bytes at the end of
// the stage's 12 KB plane tile.  Warp 6 then writes, for the group's rows
// r < R and 16-byte chunks j of the block, hi/mid/lo of those 8 values into
// rows p*32 + r (p = 0, 1, 2) of the tile, chunk j at chunk position
// j ^ (row & 7) of its 128-byte row (the 128-byte swizzle); hi = RN(a),
// mid = RN(a - hi), lo = RN(a - hi - mid), all exact.  Work item
// i = lane + 32 t is (r, j) = (i / 8, i % 8); NIT items per lane.
template <int NIT>
__device__ __forceinline__ void split_block(uint8_t* btile, int rows_in_group, int lane) {
  const int n_items = rows_in_group * (BK / 8);
  const int stg_off = B_TILE_BYTES - rows_in_group * BK * 4;
  const float* stg = reinterpret_cast<const float*>(btile + stg_off);
  float a[NIT][8];
#pragma unroll
  for (int t = 0; t < NIT; ++t) {
    const int it = lane + 32 * t;
    const int off = it < n_items ? (it >> 3) * BK + (it & 7) * 8 : 0;
    const float4 x0 = *reinterpret_cast<const float4*>(stg + off);
    const float4 x1 = *reinterpret_cast<const float4*>(stg + off + 4);
    a[t][0] = x0.x; a[t][1] = x0.y; a[t][2] = x0.z; a[t][3] = x0.w;
    a[t][4] = x1.x; a[t][5] = x1.y; a[t][6] = x1.z; a[t][7] = x1.w;
  }
  __syncwarp();      // every lane has read the staged block before any write
  // the staging area, except the group's own plane rows, back to zero
  for (int off = stg_off + lane * 16; off < B_TILE_BYTES; off += 32 * 16)
    if (((off >> 7) & (NP - 1)) >= rows_in_group)
      *reinterpret_cast<uint4*>(btile + off) = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
  for (int t = 0; t < NIT; ++t) {
    const int it = lane + 32 * t;
    if (it >= n_items) continue;
    const int r = it >> 3, j = it & 7;
    // pairs of elements, element 2i in the low half; the differences are
    // exact, so the fused multiply-add by -1 is a plain exact subtraction
    uint32_t h[4], m[4], l[4];
    const float2 neg1 = make_float2(-1.0f, -1.0f);
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      const float2 x = make_float2(a[t][e], a[t][e + 1]);
      h[e >> 1] = bf16x2_rn(x);
      const float2 r1 = __ffma2_rn(bf16x2_to_float2(h[e >> 1]), neg1, x);
      m[e >> 1] = bf16x2_rn(r1);
      const float2 r2 = __ffma2_rn(bf16x2_to_float2(m[e >> 1]), neg1, r1);
      l[e >> 1] = bf16x2_rn(r2);
    }
    const int chunk = (j ^ (r & 7)) * 16;
    *reinterpret_cast<uint4*>(btile + (0 * NP + r) * 128 + chunk) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(btile + (1 * NP + r) * 128 + chunk) = make_uint4(m[0], m[1], m[2], m[3]);
    *reinterpret_cast<uint4*>(btile + (2 * NP + r) * 128 + chunk) = make_uint4(l[0], l[1], l[2], l[3]);
  }
}

// Groups of more than 16 rows: A [R][H] fp32 -> planes [G][96][H] bf16 in
// global memory, plane p of row r of group g at plane-row p * 32 + (r - 32 g),
// rows past R zero; the same hi/mid/lo split.
__global__ void split_planes_kernel(const float* __restrict__ act, int rows, int hidden,
                                    int groups, __nv_bfloat16* __restrict__ planes) {
  // the projection that follows reads only the weights before its own
  // wait, so it may launch at once and start its weight stream; the kernels
  // after it launch only once it is past its wait
  pdl_trigger();
  pdl_wait();
  const int chunks = hidden / 8;
  const long long total = static_cast<long long>(groups) * NP * chunks;
  const float2 neg1 = make_float2(-1.0f, -1.0f);
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(i % chunks);
    const int r = static_cast<int>(i / chunks);        // global row (g * 32 + local row)
    const int g = r / NP, rl = r % NP;
    float a[8];
    const float* src = act + static_cast<size_t>(r < rows ? r : 0) * hidden + c * 8;
#pragma unroll
    for (int j = 0; j < 8; ++j) a[j] = r < rows ? src[j] : 0.0f;
    uint32_t h[4], m[4], l[4];
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      const float2 x = make_float2(a[e], a[e + 1]);
      h[e >> 1] = bf16x2_rn(x);
      const float2 r1 = __ffma2_rn(bf16x2_to_float2(h[e >> 1]), neg1, x);
      m[e >> 1] = bf16x2_rn(r1);
      const float2 r2 = __ffma2_rn(bf16x2_to_float2(m[e >> 1]), neg1, r1);
      l[e >> 1] = bf16x2_rn(r2);
    }
    const size_t base = (static_cast<size_t>(g) * BN + rl) * hidden + c * 8;
    *reinterpret_cast<uint4*>(planes + base) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(planes + base + static_cast<size_t>(NP) * hidden) =
        make_uint4(m[0], m[1], m[2], m[3]);
    *reinterpret_cast<uint4*>(planes + base + static_cast<size_t>(2 * NP) * hidden) =
        make_uint4(l[0], l[1], l[2], l[3]);
  }
}

// NIT > 0: planes built in the kernel (tm_x: the fp32 activations, boxes of
// 64 x R); NIT == 0: plane tiles loaded (tm_x: the bf16 planes of this
// group, boxes of 64 x 96, 128-byte swizzle).
template <int NIT>
__global__ void __launch_bounds__(THREADS, 1)
    project_tc_kernel(const __grid_constant__ CUtensorMap tm_w,
                      const __grid_constant__ CUtensorMap tm_x, int hidden, int vocab,
                      int rows_in_group, int row_base, float* __restrict__ logits,
                      float* __restrict__ logits2, uint32_t* __restrict__ gmax, int ngroups,
                      int32_t* status) {
  constexpr bool kFused = NIT > 0;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  // barrier slots: full[STAGES], empty[STAGES], tmem_full[2], tmem_empty[2],
  // act_full[STAGES]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 3 * STAGES + 4);
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
  auto afull_bar = [&](int s) { return smem_u32(bars + 2 * STAGES + 4 + s); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // the bytes' arrive.expect_tx, and the plane warp's arrival when it
      // builds the planes
      mbar_init(full_bar(s), kFused ? 2 : 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(afull_bar(s), 1);      // the staged activations
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
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_x)) : "memory");
  }
  if (kFused && warp == PLANE_WARP) {
    // zero every stage's plane tile once (private shared memory, so before
    // the wait below): rows past the group are never written again
    for (int s = 0; s < STAGES; ++s) {
      uint4* t = reinterpret_cast<uint4*>(smem + s * STAGE_BYTES + MT * W_TILE_BYTES);
      for (int i = lane; i < B_TILE_BYTES / 16; i += 32) t[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    // ordered before the bulk copies that later land in these tiles
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_holder)),
                 "r"(TMEM_ALLOC)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncwarp();     // lanes of warps 0 and 1 took single-lane branches above
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // No kernel of a window writes the weights, so the producer requests the
  // first stages' weight blocks before the wait: the weight stream starts
  // while the previous kernel finishes.  The stages complete only after the
  // wait, when the producer arrives on them (with the activations' bytes).
  int prefilled = 0;
  if (warp == 0 && lane == 0) {
    const uint64_t pol_w = l2_policy_evict_first();
    const int my_units =
        static_cast<int>(blockIdx.x) < n_units ? (n_units - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    prefilled = min(STAGES, my_units * n_kb);
    for (int i = 0; i < prefilled; ++i) {
      const int u = blockIdx.x + (i / n_kb) * gridDim.x;
      mbar_add_tx(full_bar(i), MT * W_TILE_BYTES);
      tma_load_2d(smem_u32(smem + i * STAGE_BYTES), &tm_w, (i % n_kb) * BK, u * MT * BM,
                  full_bar(i), pol_w);
    }
  }
  // from here on the activations and the logits buffer are touched, so wait
  // for the previous kernel to complete
  pdl_wait();
  // a window starts with this kernel: its dependents may launch only now,
  // once every kernel before the window is complete, because the later
  // kernels of the window read the window's inputs before their own wait
  pdl_trigger();

  if (warp == 0) {
    // ---------------- producer: TMA ring ----------------
    if (lane == 0) {
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_x = l2_policy_evict_last();     // shared by every CTA
      const uint32_t a_bytes = static_cast<uint32_t>(rows_in_group) * BK * 4;
      const int stg_off = B_TILE_BYTES - rows_in_group * BK * 4;
      int s = 0;
      uint32_t ph = 0;
      int it = 0;
      int last_fill_parity[STAGES];
      for (int i = 0; i < STAGES; ++i) last_fill_parity[i] = i < prefilled ? 0 : -1;
      for (int u = blockIdx.x; u < n_units && !*abort_flag; u += gridDim.x) {
        for (int kb = 0; kb < n_kb; ++kb, ++it) {
          if (!mbar_wait(empty_bar(s), ph ^ 1, abort_flag, status)) break;
          uint8_t* st = smem + s * STAGE_BYTES;
          if (kFused) {
            mbar_expect_tx(afull_bar(s), a_bytes);
            tma_load_2d(smem_u32(st + MT * W_TILE_BYTES + stg_off), &tm_x, kb * BK, row_base,
                        afull_bar(s), pol_x);
          }
          // the full box always lands: rows past the vocabulary arrive as
          // zeros; a prefilled stage's weight bytes were expected already
          const bool pre = it < prefilled;
          mbar_expect_tx(full_bar(s), (pre ? 0u : static_cast<uint32_t>(MT * W_TILE_BYTES)) +
                                          (kFused ? 0u : static_cast<uint32_t>(B_TILE_BYTES)));
          if (!kFused)
            tma_load_2d(smem_u32(st + MT * W_TILE_BYTES), &tm_x, kb * BK, 0, full_bar(s), pol_x);
          if (!pre) tma_load_2d(smem_u32(st), &tm_w, kb * BK, u * MT * BM, full_bar(s), pol_w);
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
          while (kFused &&
                 !mbar_try_wait(afull_bar(i), static_cast<uint32_t>(last_fill_parity[i])) &&
                 clock64() - t0 < kWaitLimitCycles / 8) {
          }
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
  } else if (warp == PLANE_WARP) {
    // ---------------- planes: activations -> swizzled bf16 plane tiles ----------------
    if constexpr (kFused) {
      int s = 0;
      uint32_t ph = 0;
      for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
        if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
        bool ok = true;
        for (int kb = 0; kb < n_kb; ++kb) {
          ok = mbar_wait(afull_bar(s), ph, abort_flag, status);
          if (!__all_sync(0xffffffffu, ok)) break;
          split_block<NIT>(smem + s * STAGE_BYTES + MT * W_TILE_BYTES, rows_in_group, lane);
          // generic-proxy writes, read by the MMA (async proxy) after the barrier
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) mbar_arrive(full_bar(s));
          if (++s == STAGES) {
            s = 0;
            ph ^= 1;
          }
        }
        if (!__all_sync(0xffffffffu, ok)) break;
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
              if (v < vocab) {
                const size_t at = static_cast<size_t>(row_base + r) * vocab + v;
                logits[at] = x;
                if (logits2) logits2[at] = x;     // a second copy (penalised in place later)
              }
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
  // Each role above runs on one lane of its warp (producer, MMA issuer) while
  // the other lanes come straight here, so a warp's lanes reach this point at
  // different times.  The block barrier counts arrivals per warp, so a warp
  // must arrive as a whole: without the reconvergence below the barrier was
  // measured to release while the epilogue warps were still reading TMEM,
  // and the dealloc that follows it could then free TMEM in use.
  __syncwarp();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_ALLOC)
                 : "memory");
  }
}

}  // namespace tc

// ---------------------------------------------------------------------------
// host side

namespace {
// The driver's tensor-map encoder, looked up once per process (a driver entry
// point, the same for every device); null if the driver lacks it.
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}
}  // namespace

// 2-D bf16 tensor map over a row-major [outer][inner] array, tiles of
// box_outer x box_inner elements, 128-byte swizzle (box_inner * 2 == 128).
bool encode_bf16_tile(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                      uint32_t box_inner, uint32_t box_outer) {
  const auto g_encode = encoder();
  if (!g_encode) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D fp32 tensor map for tensor stores: boxes of box_outer rows of
// box_inner floats (box_inner * 4 == 128: one 128-byte swizzled row each);
// parts of a box past the array are not written.
bool encode_f32_box_sw128(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                          uint32_t box_inner, uint32_t box_outer) {
  const auto g_encode = encoder();
  if (!g_encode) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 4};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D fp32 tensor map over a row-major [outer][inner] array, tiles of
// box_outer x box_inner elements, no swizzle; reads past the array are zero.
bool encode_f32_rows(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                     uint32_t box_inner, uint32_t box_outer) {
  const auto g_encode = encoder();
  if (!g_encode) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 4};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

template <int NIT>
cudaError_t launch_group(const CUtensorMap& tm_w, const CUtensorMap& tm_x, int hidden, int vocab,
                         int rg, int row_base, float* logits, float* logits2, uint32_t* gmax,
                         int32_t* status, int grid, cudaStream_t stream) {
  static std::atomic<bool> attr_set[kMaxDevices];
  const cudaError_t e = set_smem_limit_once(tc::project_tc_kernel<NIT>, tc::SMEM_BYTES, attr_set);
  if (e != cudaSuccess) return e;
  return launch_pdl(tc::project_tc_kernel<NIT>, dim3(grid), dim3(tc::THREADS), tc::SMEM_BYTES,
                    stream, tm_w, tm_x, hidden, vocab, rg, row_base, logits, logits2, gmax,
                    (vocab + 31) / 32, status);
}

}  // namespace

size_t tc_scratch_bytes(int rows, int hidden) {
  const size_t r = static_cast<size_t>(rows), h = static_cast<size_t>(hidden);
  if (rows <= tc::FUSED_MAX_ROWS) return r * h * sizeof(float);     // an aligned copy of act
  const size_t groups = (r + tc::NP - 1) / tc::NP;
  return groups * tc::BN * h * 2;                                   // the planes
}

namespace {

// One CTA per SM; or, when fewer CTAs take the same number of units each and
// the SMs this leaves free can hold the row sampling kernel that follows in a
// window (one CTA per row, two per SM), that smaller grid: the sampling
// kernel then sits beside the projection, and the next window's projection
// CTAs all start on SMs of their own.
int tc_grid(int rows, int vocab, int num_sms) {
  const int n_mtiles = (vocab + tc::BM - 1) / tc::BM;
  const int n_units = (n_mtiles + tc::MT - 1) / tc::MT;
  int grid = std::min(n_units, num_sms);
  const int per_cta = (n_units + num_sms - 1) / num_sms;
  const int balanced = (n_units + per_cta - 1) / per_cta;
  if ((rows + 1) / 2 <= num_sms - balanced) grid = balanced;
  return grid;
}

}  // namespace

int tc_early_free_sms(int rows, int vocab) {
  const int num_sms = device_sm_count();
  if (num_sms <= 0) return 0;
  const int grid = tc_grid(rows, vocab, num_sms);
  const int n_units = ((vocab + tc::BM - 1) / tc::BM + tc::MT - 1) / tc::MT;
  const int per_cta = (n_units + grid - 1) / grid;
  // SMs without a CTA, plus the CTAs with one unit fewer than the others
  return (num_sms - grid) + (grid * per_cta - n_units);
}

int launch_project_tc(const uint16_t* weight, const float* act, int rows, int hidden, int vocab,
                      float* logits, float* logits2, void* scratch, uint32_t* gmax,
                      int32_t* status, cudaStream_t stream) {
  const int num_sms = device_sm_count();
  if (num_sms <= 0) return VR_ERR_CUDA;
  CUtensorMap tm_w;
  // one 256-row box per unit and K block (both vocab tiles of the unit)
  if (!encode_bf16_tile(&tm_w, weight, hidden, vocab, tc::BK, tc::MT * tc::BM)) return VR_ERR_ARG;
  const int grid = tc_grid(rows, vocab, num_sms);

  if (rows <= tc::FUSED_MAX_ROWS) {
    // one group, planes built in the kernel from the activations
    if (reinterpret_cast<uintptr_t>(act) % 16) {
      // a tensor map needs a 16-byte aligned base: stage the rows in scratch
      if (cudaMemcpyAsync(scratch, act, static_cast<size_t>(rows) * hidden * sizeof(float),
                          cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
        return VR_ERR_CUDA;
      act = static_cast<const float*>(scratch);
    }
    CUtensorMap tm_a;
    if (!encode_f32_rows(&tm_a, act, hidden, rows, tc::BK, rows)) return VR_ERR_ARG;
    // plane items per lane of the plane warp: rows x 8 chunks over 32 lanes
    const int nit = (rows * (tc::BK / 8) + 31) / 32;
    cudaError_t e;
    if (nit <= 1)
      e = launch_group<1>(tm_w, tm_a, hidden, vocab, rows, 0, logits, logits2, gmax, status, grid,
                          stream);
    else if (nit <= 2)
      e = launch_group<2>(tm_w, tm_a, hidden, vocab, rows, 0, logits, logits2, gmax, status, grid,
                          stream);
    else
      e = launch_group<4>(tm_w, tm_a, hidden, vocab, rows, 0, logits, logits2, gmax, status, grid,
                          stream);
    if (e != cudaSuccess) return VR_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? VR_OK : VR_ERR_CUDA;
  }

  // groups of 32 rows, planes written by the split kernel first
  const int groups = (rows + tc::NP - 1) / tc::NP;
  auto* pl = static_cast<__nv_bfloat16*>(scratch);
  {
    const long long work = static_cast<long long>(groups) * tc::NP * (hidden / 8);
    const int threads = 256;
    const int blocks = static_cast<int>(std::min<long long>((work + threads - 1) / threads,
                                                            static_cast<long long>(num_sms) * 8));
    if (launch_pdl(tc::split_planes_kernel, dim3(blocks), dim3(threads), 0, stream, act, rows,
                   hidden, groups, pl) != cudaSuccess)
      return VR_ERR_CUDA;
  }
  for (int g = 0; g < groups; ++g) {
    CUtensorMap tm_b;
    if (!encode_bf16_tile(&tm_b, pl + static_cast<size_t>(g) * tc::BN * hidden, hidden, tc::BN,
                          tc::BK, tc::BN))
      return VR_ERR_ARG;
    const int rg = std::min(tc::NP, rows - g * tc::NP);
    if (launch_group<0>(tm_w, tm_b, hidden, vocab, rg, g * tc::NP, logits, logits2, gmax, status,
                        grid, stream) != cudaSuccess)
      return VR_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? VR_OK : VR_ERR_CUDA;
}

}  // namespace vr
