// Newton-Schulz phase GEMM on tcgen05 with CTA pairs (cta_group::2).
//
// Same phases, problems and epilogues as k_ns_tc.cu ("架构设计" §1: A = X X^T,
// B = b A + c A A, X <- a X + B X), but each output tile is 256 x 256 and is
// computed by a cluster of two CTAs on two SMs:
//   * CTA r of the pair loads rows [128r, 128r+128) of the tile's A operand
//     and columns [128r, 128r+128) of its B operand (K-contiguous: one
//     64 x 128 TMA box; M/N-contiguous: two 64 x 64 boxes) into its own
//     4-stage shared-memory ring, and the completion of both CTAs' copies is counted on
//     the leader CTA's `full` barrier;
//   * one thread of the leader (rank 0) issues tcgen05.mma.cta_group::2
//     with M = 256, N = 256, K = 16: the tensor cores read A from both CTAs
//     and B from both CTAs, and each CTA's TMEM receives its own 128 rows of
//     the fp32 accumulator;
//   * tcgen05.commit with a two-CTA multicast frees the ring slot in both
//     CTAs and hands the accumulator to both CTAs' epilogue warps, which run
//     the shared fused epilogue on their own 128 rows and then arrive on the
//     leader's `tempty` barrier (one arrival per epilogue warp of both CTAs).
// Per SM and per 16-deep k-step the operands are 128 x 16 of A and 128 x 16
// of B (8 KiB) for 128 x 256 x 16 multiply-adds, against 12 KiB in the
// one-CTA kernel: two thirds of the shared-memory fill and L2 read traffic
// per flop.
//
// Symmetric outputs (A = X X^T, B = b A + c A A) keep only their 256-blocks
// on or above the diagonal: nothing is mirrored.  Where a later product reads
// such a matrix as an operand, a k-block that falls below the diagonal is
// loaded from the transposed stored block as an M/N-contiguous tile, and the
// MMA descriptor for that k-block says so (NsProblem::tri).
//
// Wide tiles (the WIDE instantiation): a tile may instead be 256 x 512, two
// adjacent 256-column blocks that share the A rows.  Per k-block each CTA
// then loads 128 rows of A and 2 x 128 rows of B (48 KiB, 3-stage ring) and
// the leader issues two MMAs into two 256-column accumulators: 1.5x the
// operand bytes for 2x the multiply-adds.  Measured, that pays only where
// the main loop is long (the Gram of the large classes: a few per cent);
// the host picks the launches.  The two accumulators fill all
// 512 TMEM columns, so a wide tile is not double-buffered against the next
// one; the accumulator "slots" (column halves) are handed out in sequence
// (a narrow tile takes one, a wide tile two), and each slot has its own
// full/empty barriers.  In a wide tile the 4 epilogue warps of column half
// h drain slot h's 256 columns and arrive twice on its empty barrier, so
// every slot use still counts 16 arrivals.
//
// Every spin-wait is bounded; on a timeout the CTA records the error, stops
// issuing, and both CTAs meet at the final cluster barrier before the pair
// frees its TMEM.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"
#include "ns_epilogue.cuh"
#include "ptx.cuh"

namespace dmuon {
namespace {

constexpr int TILE = kTc2Tile;  // 256 x 256 per CTA pair
constexpr int BK = 64;
constexpr uint32_t HALF_BYTES = 128 * BK * 2;         // 16 KiB: 128 rows x 64 k, bf16
template <bool WIDE>
__host__ __device__ constexpr uint32_t stage_bytes() {
  return (WIDE ? 3 : 2) * HALF_BYTES;  // A half + one (or two) B halves per CTA
}
constexpr uint32_t MN_BOX_BYTES = 64 * 64 * 2;        // 8 KiB
// Warps: 0 A producer, 1 MMA, 2 .. 2+EPI-1 epilogue, 2+EPI B producer.  The
// epilogue has EPI = 4 warps (one per TMEM lane quarter) or 8 (two per lane
// quarter, each on half of the tile's columns).  Eight drain a tile twice as
// fast, which pays where the main loop is short (K of a few k-blocks: small
// matrices), but their global loads then compete with the operand copies
// for each SM's memory bandwidth, which slows long main loops; the host
// picks per launch.  The fused update always runs with 4 (its staging boxes
// and registers leave no room for more warps).
template <int EPI>
constexpr int threads_of() {
  return (3 + EPI) * 32;
}
constexpr uint32_t kTmemCols = 512;
// Epilogue staging per warp: 2 boxes of 32 x 64 bf16; the fused update
// stages kFusedWBoxes fp32 boxes of 32 x 32 (W, loaded and stored by TMA)
// and 2 bf16 boxes of 32 x 64 (param).
template <bool FUSE>
__host__ __device__ constexpr uint32_t staging_per_warp() {
  return FUSE ? (kFusedWBoxes + 2) * 4096 : 2 * 4096;
}
// mbarriers: full/empty per ring stage, 2 accumulator full/empty pairs, the
// drain barrier, and (fused update) one per W box buffer of each epilogue warp.
template <int STAGES, int EPI, bool FUSE>
__host__ __device__ constexpr int num_bars() {
  return 2 * STAGES + 2 + 2 + 1 + (FUSE ? kFusedWBoxes * EPI : 0);
}
template <int STAGES, int EPI, bool WIDE = false, bool FUSE = false>
constexpr size_t smem_bytes() {
  return 1024 + STAGES * stage_bytes<WIDE>() + EPI * staging_per_warp<FUSE>() + num_bars<STAGES, EPI, FUSE>() * 8 +
         16;
}
static_assert(smem_bytes<5, 8>() <= 227 * 1024, "shared memory budget");
// The fused update runs with a 4-stage ring: a fifth stage does not fit
// beside its W boxes.
static_assert(smem_bytes<4, 4, false, true>() <= 227 * 1024, "shared memory budget (fused update)");
// 3 stages of 48 KiB: a fourth does not fit beside 8 warps' staging boxes.
static_assert(smem_bytes<3, 8, true>() <= 227 * 1024, "shared memory budget (wide)");
// Every CTA allocates all 512 TMEM columns, so two CTAs must never share an
// SM: a second resident pair could hold one SM's TMEM while its partner waits
// for the other's.  Asking for more than half of the SM's 228 KiB of shared
// memory rules that out.
static_assert(smem_bytes<4, 4>() > 114 * 1024, "one CTA per SM");

__device__ __forceinline__ uint64_t desc_k(uint32_t base, int kk) {
  return smem_desc_sw128(base + 32u * kk, 16u, 1024u);
}
__device__ __forceinline__ uint64_t desc_mn(uint32_t base, int kk) {
  return smem_desc_sw128(base + 2048u * kk, MN_BOX_BYTES, 1024u);
}

// What the producer and the MMA issuer need of one tile.  Loaded one tile
// ahead, so the dependent global loads (tile list, then problem) overlap the
// previous tile's main loop instead of stalling the pipeline between tiles.
struct TileInfo {
  int m0, n0;  // tile origin (rows, columns) of the pair
  int map_a, map_b, z, majors, nk;
  int tri, map_a_t, map_b_t;
  int wide;    // 1: 256 x 512 (two column blocks)
};

__device__ __forceinline__ TileInfo load_tile_info(const NsLaunch& L, int t) {
  const uint2 tile = L.tiles[t];
  const NsProblem& P = L.probs[tile.x & kTileProbMask];
  TileInfo I;
  I.m0 = static_cast<int>(tile.y >> 16) * TILE;
  I.n0 = static_cast<int>(tile.y & 0xFFFFu) * TILE;
  I.wide = (tile.x & kTileWideBit) ? 1 : 0;
  I.map_a = P.map_a;
  I.map_b = P.map_b;
  I.z = P.z;
  I.majors = P.majors;
  I.nk = (P.K + BK - 1) / BK;
  I.tri = L.tri ? P.tri : 0;
  I.map_a_t = P.map_a_t;
  I.map_b_t = P.map_b_t;
  return I;
}

// A k-block of a symmetric operand stored as upper 256-blocks only: below
// the diagonal (k-block before the operand's row block) it is read from the
// transposed stored block, M/N-contiguous.
__device__ __forceinline__ bool tri_below(int tri_bit, int k0, int row0) {
  return tri_bit && (k0 >> 8) < (row0 >> 8);
}

// FUSE: the last Combine, which applies the update instead of storing X.
// WIDE: the tile list may hold 256 x 512 tiles.
// PIPE: the launch reads no aux operand, and the epilogue drains TMEM with
// the next chunk's load in flight (ns_epilogue_tile_staged_pipe).
template <int STAGES, bool FUSE, int EPI, bool WIDE = false, bool PIPE = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(threads_of<EPI>(), 1)
    ns_tc2_kernel(const NsLaunch L) {
  static_assert(EPI == 4 || (EPI == 8 && !FUSE), "epilogue warp count");
  static_assert(!WIDE || (EPI == 8 && !FUSE), "wide tiles: 8 epilogue warps, no fused update");
  static_assert(!PIPE || !FUSE, "pipelined drain: plain stores only");
  constexpr uint32_t STAGE_BYTES = stage_bytes<WIDE>();
  constexpr int kProducerBWarp = 2 + EPI;
  constexpr int kNumBars = num_bars<STAGES, EPI, FUSE>();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t ring = smem_u32(smem);
  const uint32_t staging = ring + STAGES * STAGE_BYTES;  // 1 KiB aligned (swizzled TMA source)
  constexpr uint32_t kStaging = staging_per_warp<FUSE>();
  uint64_t* bar_mem = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES + EPI * kStaging);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_mem + kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const uint32_t bar0 = smem_u32(bar_mem);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
  auto tempty = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
  const uint32_t drain = bar0 + 8u * (2 * STAGES + 4);
  const uint32_t wbars = bar0 + 8u * (2 * STAGES + 5);  // fused update: kFusedWBoxes per epilogue warp

  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), 2);  // one arrival per operand producer (leader)
      mbar_init(empty(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull(a), 1);
      mbar_init(tempty(a), 2 * EPI);  // every epilogue warp of both CTAs
    }
    mbar_init(drain, 1);
    for (int i = 0; i < (FUSE ? kFusedWBoxes * EPI : 0); ++i) mbar_init(wbars + 8u * i, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers exist before any cross-CTA signal
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int t_begin = L.cta_begin[pair];
  const int t_end = L.cta_begin[pair + 1];

  if ((warp == 0 || warp == kProducerBWarp) && lane == 0) {
    // ------------------------------------------- producers (A: warp 0, B: warp 6)
    // Each operand has its own issuing thread, so the TMA issue work of a
    // k-block is split over two warps.  Both follow the same ring and wait on
    // the same `empty` barriers; in the leader each arms `full` with the bytes
    // of its operand for both CTAs (the barrier takes two arrivals).
    const int which = (warp == 0) ? 0 : 1;
    const uint32_t dst_off = which ? HALF_BYTES : 0u;
    int stage = 0;
    uint32_t phase = 0;
    int fills[STAGES] = {};
    bool ok = true;
    TileInfo cur{}, nxt{};
    if (t_begin < t_end) cur = load_tile_info(L, t_begin);
    for (int t = t_begin; t < t_end && ok; ++t) {
      if (t + 1 < t_end) nxt = load_tile_info(L, t + 1);
      const int tile_row0 = which ? cur.n0 : cur.m0;
      const CUtensorMap* map = L.maps + (which ? cur.map_b : cur.map_a);
      const CUtensorMap* map_t = L.maps + (which ? cur.map_b_t : cur.map_a_t);
      const bool mn = ((cur.majors >> which) & 1) != 0;
      const bool tri = ((cur.tri >> which) & 1) != 0;
      const int z = cur.z;
      const int nk = cur.nk;
      // B of a wide tile: two 256-row blocks of the operand.
      const int nsub = (WIDE && which && cur.wide) ? 2 : 1;
      cur = nxt;
      for (int kb = 0; kb < nk; ++kb) {
        if (!mbar_wait_bounded_cluster(empty(stage), phase ^ 1u, abort_flag, L.err, kErrTimeoutProducer)) {
          ok = false;
          break;
        }
        const uint32_t leader_full = mapa_shared(full(stage), 0);
        if (leader) mbar_expect_tx(full(stage), 2 * HALF_BYTES * static_cast<uint32_t>(nsub));
        ++fills[stage];
        const int k0 = kb * BK;
        for (int h = 0; h < nsub; ++h) {
          const int blk_row0 = tile_row0 + TILE * h;
          const int row0 = blk_row0 + 128 * static_cast<int>(rank);
          const uint32_t dst = ring + stage * STAGE_BYTES + dst_off + static_cast<uint32_t>(h) * HALF_BYTES;
          // k-blocks before the operand block's diagonal block come transposed.
          if (tri && (k0 >> 8) < (blk_row0 >> 8)) {
            tma_load_3d_pair(dst, map_t, leader_full, row0, k0, z);
            tma_load_3d_pair(dst + MN_BOX_BYTES, map_t, leader_full, row0 + 64, k0, z);
          } else if (!mn) {
            tma_load_3d_pair(dst, map, leader_full, k0, row0, z);
          } else {
            tma_load_3d_pair(dst, map, leader_full, row0, k0, z);
            tma_load_3d_pair(dst + MN_BOX_BYTES, map, leader_full, row0 + 64, k0, z);
          }
        }
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok && leader) {
      // The leader's barrier counts both CTAs' bytes: let every armed phase
      // land before the pair tears down.
      for (int s = 0; s < STAGES; ++s) {
        if (fills[s] > 0) {
          volatile int no_abort = 0;
          mbar_wait_bounded_cluster(full(s), static_cast<uint32_t>(fills[s] - 1) & 1u, &no_abort, nullptr, 0,
                                    100000000ull);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------- MMA issuer (leader only)
    if (leader && lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int use = 0;  // accumulator slot uses so far (slot = use & 1)
      TileInfo cur{}, nxt{};
      if (t_begin < t_end) cur = load_tile_info(L, t_begin);
      for (int t = t_begin; t < t_end && ok; ++t) {
        if (t + 1 < t_end) nxt = load_tile_info(L, t + 1);
        const bool a_mn = (cur.majors & 1) != 0;
        const bool b_mn = (cur.majors & 2) != 0;
        const int tri = cur.tri;
        const int tile_m0 = cur.m0, tile_n0 = cur.n0;
        const int nk = cur.nk;
        const int nsub = (WIDE && cur.wide) ? 2 : 1;
        cur = nxt;
        for (int h = 0; h < nsub && ok; ++h) {
          const int u = use + h;
          if (!mbar_wait_bounded_cluster(tempty(u & 1), (static_cast<uint32_t>(u >> 1) & 1u) ^ 1u, abort_flag, L.err,
                                         kErrTimeoutMma))
            ok = false;
        }
        if (!ok) break;
        tc_fence_after();
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait_bounded_cluster(full(stage), phase, abort_flag, L.err, kErrTimeoutMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = ring + stage * STAGE_BYTES;
          const bool a_is_mn = a_mn || tri_below(tri & 1, kb * BK, tile_m0);
          if (nsub == 1) {
            const uint32_t sb = sa + HALF_BYTES;
            const bool b_is_mn = b_mn || tri_below(tri & 2, kb * BK, tile_n0);
            const uint32_t idesc = idesc_bf16_f32(TILE, TILE, a_is_mn, b_is_mn);
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>((use & 1) * TILE);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              const uint64_t ad = a_is_mn ? desc_mn(sa, kk) : desc_k(sa, kk);
              const uint64_t bd = b_is_mn ? desc_mn(sb, kk) : desc_k(sb, kk);
              umma_bf16_pair(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
            }
          } else {
            // Both column halves per 16-deep k-step, the second taking A
            // from the collector buffer the first filled.
            const uint32_t sb0 = sa + HALF_BYTES, sb1 = sa + 2 * HALF_BYTES;
            const bool b0_mn = b_mn || tri_below(tri & 2, kb * BK, tile_n0);
            const bool b1_mn = b_mn || tri_below(tri & 2, kb * BK, tile_n0 + TILE);
            const uint32_t idesc0 = idesc_bf16_f32(TILE, TILE, a_is_mn, b0_mn);
            const uint32_t idesc1 = idesc_bf16_f32(TILE, TILE, a_is_mn, b1_mn);
            const uint32_t d0 = tmem_base + static_cast<uint32_t>((use & 1) * TILE);
            const uint32_t d1 = tmem_base + static_cast<uint32_t>(((use + 1) & 1) * TILE);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              const uint64_t ad = a_is_mn ? desc_mn(sa, kk) : desc_k(sa, kk);
              const uint64_t bd0 = b0_mn ? desc_mn(sb0, kk) : desc_k(sb0, kk);
              const uint64_t bd1 = b1_mn ? desc_mn(sb1, kk) : desc_k(sb1, kk);
              const uint32_t acc = (kb | kk) != 0 ? 1u : 0u;
              umma_bf16_pair_a_fill(d0, ad, bd0, idesc0, acc);
              umma_bf16_pair_a_lastuse(d1, ad, bd1, idesc1, acc);
            }
          }
          umma_commit_pair_multicast(empty(stage), 0x3);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok)
          for (int h = 0; h < nsub; ++h) umma_commit_pair_multicast(tfull((use + h) & 1), 0x3);
        use += nsub;
      }
      umma_commit_pair_multicast(drain, 0x1);
      volatile int no_abort = 0;
      mbar_wait_bounded_cluster(drain, 0, &no_abort, L.err, kErrTimeoutDrain);
    }
  } else if (warp >= 2 && warp < 2 + EPI) {
    // ------------------------------------------------------------ epilogue
    // A warp reaches the TMEM lanes of its warp index mod 4; with 8 warps
    // the two warps of one lane quarter take one column half each.
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row_in_tile = 128 * static_cast<int>(rank) + quarter * 32 + lane;
    const uint32_t my_staging = staging + static_cast<uint32_t>(warp - 2) * kStaging;
    uint32_t box_count = 0;
    const uint32_t my_wbars = wbars + 8u * static_cast<uint32_t>(kFusedWBoxes * (warp - 2));
    uint32_t w_issued = 0, w_used = 0;  // fused update: W boxes requested / consumed
    int use = 0;  // accumulator slot uses so far, as counted by the MMA issuer
    for (int t = t_begin; t < t_end; ++t) {
      const uint2 tile = L.tiles[t];
      const NsProblem& P = L.probs[tile.x & kTileProbMask];
      const int tm = static_cast<int>(tile.y >> 16), tn = static_cast<int>(tile.y & 0xFFFFu);
      const bool wide = WIDE && (tile.x & kTileWideBit) != 0;
      // Narrow tile: every warp drains its column window of the one slot.
      // Wide tile: the warps of column half h drain all 256 columns of slot
      // (use + h), i.e. column block tn + h of the output.
      const int u = wide ? use + half : use;
      const int acc = u & 1;
      const uint32_t acc_phase = static_cast<uint32_t>(u >> 1) & 1u;
      const int sub_tn = wide ? tn + half : tn;
      const int c_begin = (EPI == 8 && !wide) ? 4 * half : 0;
      const int c_end = (EPI == 8 && !wide) ? c_begin + 4 : 8;
      use += wide ? 2 : 1;
      if (FUSE) fused_w_prefetch(L, P, tm * TILE, sub_tn * TILE, row_in_tile, my_staging, my_wbars, w_issued);
      if (!mbar_wait_bounded_cluster(tfull(acc), acc_phase, abort_flag, L.err, kErrTimeoutEpilogue)) break;
      tc_fence_after();
      const uint32_t t_lane =
          tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * TILE);
      if (FUSE) {
        if (!ns_epilogue_tile_fused_tma(L, P, tm * TILE, sub_tn * TILE, row_in_tile, t_lane, my_staging, my_wbars,
                                        w_issued, w_used, abort_flag))
          break;
      } else if (PIPE)
        ns_epilogue_tile_staged_pipe(L, P, tm * TILE, sub_tn * TILE, row_in_tile, t_lane, my_staging, box_count,
                                     c_begin, c_end);
      else
        ns_epilogue_tile_staged(L, P, tm * TILE, sub_tn * TILE, row_in_tile, t_lane, !L.tri && P.sym && tm < sub_tn,
                                my_staging, box_count, c_begin, c_end);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        // A wide tile's slot is drained by half of the warps: each arrives
        // twice, so the slot's empty barrier completes on the same count.
        const int arrivals = wide ? 2 : 1;
        for (int i = 0; i < arrivals; ++i) {
          if (leader)
            mbar_arrive(tempty(acc));
          else
            mbar_arrive_cluster(mapa_shared(tempty(acc), 0));
        }
      }
    }
    if (FUSE) {
      // After an abort, W boxes may still be on their way into shared
      // memory: wait (bounded) for each before the block exits.
      volatile int no_abort = 0;
      for (uint32_t g = w_used; g < w_issued; ++g)
        mbar_wait_bounded(my_wbars + 8u * (g % kFusedWBoxes), (g / kFusedWBoxes) & 1u, &no_abort, nullptr, 0);
    }
    if (lane == 0) bulk_wait_group<0>();  // staged TMA stores complete
    __syncwarp();
  }

  tc_fence_before();
  cluster_sync_all();  // all MMAs drained, no more cross-CTA traffic
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

}  // namespace

template <int STAGES, bool FUSE, int EPI, bool WIDE = false, bool PIPE = false>
static cudaError_t launch_variant3(const NsLaunch& L, int n_pairs, cudaStream_t st) {
  static unsigned long long attr_mask = 0;
  constexpr size_t smem = smem_bytes<STAGES, EPI, WIDE, FUSE>();
  if (attr_needed_on_current_device(&attr_mask)) {
    cudaError_t e = cudaFuncSetAttribute(ns_tc2_kernel<STAGES, FUSE, EPI, WIDE, PIPE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_note_current_device(&attr_mask);
  }
  ns_tc2_kernel<STAGES, FUSE, EPI, WIDE, PIPE><<<2 * n_pairs, threads_of<EPI>(), smem, st>>>(L);
  return cudaGetLastError();
}

// The fused update keeps 4 epilogue warps and a 4-stage ring: on long main
// loops more concurrent W traffic slows the operand copies (measured +5 ms
// per Llama-3-8B step with 8 warps and an aux-free epilogue), and its W
// boxes leave no shared memory for more warps' staging or a fifth stage.
template <int STAGES>
static cudaError_t launch_variant(const NsLaunch& L, int n_pairs, cudaStream_t st) {
  if (L.fuse_update) return launch_variant3<4, true, 4>(L, n_pairs, st);
  // Short main loops (8 epilogue warps) are bound by the epilogue drain: a
  // launch without aux takes the pipelined drain there (GPT-2 and
  // many-small sets -2 to -3 %).  Long main loops keep the plain drain (the
  // overlapped epilogues' faster stores slowed the operand copies: +1 ms on
  // the Llama-3-8B Combine).
  const bool no_aux = L.kind == kGram || (L.kind == kCombine && L.a == 0.f);
  if (L.epi8 && no_aux && L.tri) return launch_variant3<STAGES, false, 8, false, true>(L, n_pairs, st);
  return L.epi8 ? launch_variant3<STAGES, false, 8>(L, n_pairs, st) : launch_variant3<STAGES, false, 4>(L, n_pairs, st);
}

cudaError_t launch_ns_tc2(const NsLaunch& L, int n_pairs, cudaStream_t st) {
  if (n_pairs <= 0) return cudaSuccess;
  if (L.wide) {
    if (L.fuse_update || !L.tri) return cudaErrorInvalidValue;  // not built for these
    // No aux operand: the Gram, and a Combine whose a*X is folded into B.
    const bool no_aux = L.kind == kGram || (L.kind == kCombine && L.a == 0.f);
    return no_aux ? launch_variant3<3, false, 8, true, true>(L, n_pairs, st)
                  : launch_variant3<3, false, 8, true>(L, n_pairs, st);
  }
  return (L.stages == 5) ? launch_variant<5>(L, n_pairs, st) : launch_variant<4>(L, n_pairs, st);
}

// Largest number of CTA pairs of this kernel that can be resident at once.
int ns_tc2_max_pairs() {
  static int cached = -1;
  if (cached >= 0) return cached;
  constexpr size_t smem = smem_bytes<5, 8>();
  if (cudaFuncSetAttribute(ns_tc2_kernel<5, false, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess) {
    cudaGetLastError();
    return cached = 0;
  }
  cudaLaunchConfig_t cfg = {};  // cluster shape comes from __cluster_dims__
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(threads_of<8>(), 1, 1);
  cfg.dynamicSmemBytes = smem;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, ns_tc2_kernel<5, false, 8>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  return cached = n;
}

}  // namespace dmuon
