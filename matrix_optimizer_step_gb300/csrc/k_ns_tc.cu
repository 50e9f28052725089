// Newton-Schulz phase GEMM on the 5th-generation tensor cores (tcgen05).
//
// One launch runs one phase of one NS iteration for every slice of every
// Muon tensor ("架构设计" §1: X <- aX + bXX^T X + cX(X^T X)^2, computed as
// A = X X^T, B = b A + c A A, X <- a X + B X).  Work is a flat list of
// 128 x 256 output tiles over all problems; a persistent grid of one CTA per
// SM walks its own LPT-balanced slice of that list.
//
// CTA layout (192 threads, one CTA per SM):
//   warp 0      TMA producer: one elected thread streams 128x64 A_op and
//               256x64 B_op bf16 tiles into a STAGES-deep shared-memory ring
//               (128-byte swizzle), signalling `full[s]` with tx-counts.
//   warp 1      MMA issuer: allocates 512 TMEM columns (two 128x256 fp32
//               accumulators), one thread issues tcgen05.mma (M=128, N=256,
//               K=16) per 16-wide k-step, frees ring slots with
//               tcgen05.commit -> `empty[s]`, and hands a finished
//               accumulator to the epilogue with tcgen05.commit -> `tfull[a]`.
//   warps 2..5  epilogue: each warp owns one 32-lane quarter of TMEM
//               (warp % 4), reads its rows 32 columns at a time with
//               tcgen05.ld, applies the phase's fused epilogue (scale;
//               b*A + c*acc; a*X + acc) and stores bf16 (plus the bf16
//               remainder where the problem asks for one) to global memory, then
//               releases the accumulator (`tempty[a]`).
// The two accumulators let the epilogue of tile i overlap the main loop of
// tile i+1.
//
// X X^T and B = b A + c A A are symmetric: for them only the 256 x 256
// blocks on or above the diagonal are computed (two 128-row tiles per
// block) and the epilogue of an off-diagonal block also stores its transpose
// (NsProblem::sym), which removes close to half of those two phases' work.
//
// Operand layouts: a K-contiguous operand tile is one TMA box of
// 64 (k) x rows; an M/N-contiguous operand tile is a row of boxes of
// 64 (m or n) x 64 (k).  With the 128-byte swizzle both are the canonical
// SW128 layouts of the UMMA shared-memory descriptor: K-major
// (SBO = 1024 B between 8-row groups) and MN-major (LBO = 8 KiB between
// 64-element MN blocks, SBO = 1024 B between 8-row k groups).
//
// All waits are bounded (ptx.cuh); on a timeout the CTA records an error,
// stops issuing, drains its own tensor-core work and frees TMEM before
// returning.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"
#include "ns_epilogue.cuh"
#include "ptx.cuh"

namespace dmuon {
namespace {

constexpr int BM = kTcBM, BN = kTcBN, BK = kTcBK;
constexpr int STAGES = 4;
constexpr uint32_t A_BYTES = BM * BK * 2;          // 16 KiB
constexpr uint32_t B_BYTES = BN * BK * 2;          // 32 KiB
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t MN_BOX_BYTES = 64 * 64 * 2;     // one 64x64 bf16 box, 8 KiB
constexpr uint32_t K_BOX_BYTES = 128 * 64 * 2;     // one 64x128 bf16 box, 16 KiB
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr int kNumBars = 2 * STAGES + 2 + 2 + 1;   // full, empty, tfull, tempty, drain
constexpr size_t kSmemBytes = 1024 + STAGES * STAGE_BYTES + kNumBars * 8 + 16;

static_assert(BM == 128 && BN == 256 && BK == 64, "tile geometry is hard-wired below");
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

struct Bars {
  uint32_t full, empty, tfull, tempty, drain;  // base addresses (shared::cta)
  __device__ uint32_t f(int s) const { return full + 8u * s; }
  __device__ uint32_t e(int s) const { return empty + 8u * s; }
  __device__ uint32_t tf(int a) const { return tfull + 8u * a; }
  __device__ uint32_t te(int a) const { return tempty + 8u * a; }
};

__device__ __forceinline__ void decode_tile(uint2 t, int& m0, int& n0) {
  m0 = static_cast<int>(t.y >> 16) * BM;
  n0 = static_cast<int>(t.y & 0xFFFFu) * BN;
}

// K-major SW128 operand: rows of 128 bytes, 8-row groups 1024 B apart.
// Advancing k by 16 elements moves the start address by 32 bytes.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t base, int kk) {
  return smem_desc_sw128(base + 32u * kk, 16u, 1024u);
}
// MN-major SW128 operand: 64-element MN blocks 8 KiB apart (LBO), 8-row k
// groups 1024 B apart (SBO).  Advancing k by 16 rows moves 2048 bytes.
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t base, int kk) {
  return smem_desc_sw128(base + 2048u * kk, MN_BOX_BYTES, 1024u);
}

template <bool FUSE>
__global__ void __launch_bounds__(kThreads, 1) ns_tc_kernel(const NsLaunch L) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t ring = smem_u32(smem);
  uint64_t* bar_mem = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_mem + kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  Bars bars;
  bars.full = smem_u32(bar_mem);
  bars.empty = bars.full + 8u * STAGES;
  bars.tfull = bars.empty + 8u * STAGES;
  bars.tempty = bars.tfull + 16u;
  bars.drain = bars.tempty + 16u;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bars.f(s), 1);
      mbar_init(bars.e(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bars.tf(a), 1);
      mbar_init(bars.te(a), 4);
    }
    mbar_init(bars.drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int t_begin = L.cta_begin[blockIdx.x];
  const int t_end = L.cta_begin[blockIdx.x + 1];

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int fills[STAGES] = {0, 0, 0, 0};
      bool ok = true;
      for (int t = t_begin; t < t_end && ok; ++t) {
        const uint2 tile = L.tiles[t];
        const NsProblem& P = L.probs[tile.x];
        int m0, n0;
        decode_tile(tile, m0, n0);
        const CUtensorMap* ma = L.maps + P.map_a;
        const CUtensorMap* mb = L.maps + P.map_b;
        const bool a_mn = (P.majors & 1) != 0;
        const bool b_mn = (P.majors & 2) != 0;
        const int z = P.z;
        const int nk = (P.K + BK - 1) / BK;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait_bounded(bars.e(stage), phase ^ 1u, abort_flag, L.err,
                                 kErrTimeoutProducer)) {
            ok = false;
            break;
          }
          const uint32_t full = bars.f(stage);
          mbar_expect_tx(full, STAGE_BYTES);
          ++fills[stage];
          const uint32_t sa = ring + stage * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
          const int k0 = kb * BK;
          if (!a_mn) {
            tma_load_3d(sa, ma, full, k0, m0, z);
          } else {
            tma_load_3d(sa, ma, full, m0, k0, z);
            tma_load_3d(sa + MN_BOX_BYTES, ma, full, m0 + 64, k0, z);
          }
          if (!b_mn) {
            tma_load_3d(sb, mb, full, k0, n0, z);
            tma_load_3d(sb + K_BOX_BYTES, mb, full, k0, n0 + 128, z);
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) tma_load_3d(sb + i * MN_BOX_BYTES, mb, full, n0 + 64 * i, k0, z);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Let every copy this thread issued land before the CTA exits.
        for (int s = 0; s < STAGES; ++s) {
          if (fills[s] > 0) {
            volatile int no_abort = 0;
            mbar_wait_bounded(bars.f(s), static_cast<uint32_t>(fills[s] - 1) & 1u, &no_abort,
                              nullptr, 0, 100000000ull);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int local = 0;
      for (int t = t_begin; t < t_end && ok; ++t, ++local) {
        const uint2 tile = L.tiles[t];
        const NsProblem& P = L.probs[tile.x];
        const bool a_mn = (P.majors & 1) != 0;
        const bool b_mn = (P.majors & 2) != 0;
        const uint32_t idesc = idesc_bf16_f32(BM, BN, a_mn, b_mn);
        const int nk = (P.K + BK - 1) / BK;
        const int acc = local & 1;
        const uint32_t acc_phase = static_cast<uint32_t>(local >> 1) & 1u;
        if (!mbar_wait_bounded(bars.te(acc), acc_phase ^ 1u, abort_flag, L.err, kErrTimeoutMma)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait_bounded(bars.f(stage), phase, abort_flag, L.err, kErrTimeoutMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = ring + stage * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = a_mn ? desc_mnmajor(sa, kk) : desc_kmajor(sa, kk);
            const uint64_t bd = b_mn ? desc_mnmajor(sb, kk) : desc_kmajor(sb, kk);
            umma_bf16(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          umma_commit(bars.e(stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) umma_commit(bars.tf(acc));
      }
      // Every MMA this thread issued completes before TMEM is released.
      umma_commit(bars.drain);
      volatile int no_abort = 0;
      mbar_wait_bounded(bars.drain, 0, &no_abort, L.err, kErrTimeoutDrain);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int row_in_tile = quarter * 32 + lane;
    int local = 0;
    for (int t = t_begin; t < t_end; ++t, ++local) {
      const uint2 tile = L.tiles[t];
      const NsProblem& P = L.probs[tile.x];
      int m0, n0;
      decode_tile(tile, m0, n0);
      const int acc = local & 1;
      const uint32_t acc_phase = static_cast<uint32_t>(local >> 1) & 1u;
      if (!mbar_wait_bounded(bars.tf(acc), acc_phase, abort_flag, L.err, kErrTimeoutEpilogue))
        break;
      tc_fence_after();

      const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                              static_cast<uint32_t>(acc * BN);
      ns_epilogue_tile<FUSE>(L, P, m0, n0, row_in_tile, t_lane, !FUSE && P.sym && ((m0 >> 8) < (n0 >> 8)));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.te(acc));
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace

template <bool FUSE>
static cudaError_t launch_tc_variant(const NsLaunch& L, int n_ctas, cudaStream_t st) {
  static unsigned long long attr_mask = 0;
  if (attr_needed_on_current_device(&attr_mask)) {
    cudaError_t e = cudaFuncSetAttribute(ns_tc_kernel<FUSE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    attr_note_current_device(&attr_mask);
  }
  ns_tc_kernel<FUSE><<<n_ctas, kThreads, kSmemBytes, st>>>(L);
  return cudaGetLastError();
}

cudaError_t launch_ns_tc(const NsLaunch& L, int n_ctas, cudaStream_t st) {
  if (n_ctas <= 0) return cudaSuccess;
  return L.fuse_update ? launch_tc_variant<true>(L, n_ctas, st) : launch_tc_variant<false>(L, n_ctas, st);
}

}  // namespace dmuon
