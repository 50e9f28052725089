// Fused epilogue of one Newton-Schulz output tile, shared by the one-CTA and
// the CTA-pair tcgen05 kernels.  One epilogue warp drains its 32 TMEM lanes
// (rows) of the accumulator, 32 columns at a time, applies the phase's
// epilogue (see NsKind) and stores bf16 (plus, in the first iterations, the
// bf16 remainder v - bf16(v), and the transposed copy of a symmetric
// off-diagonal block where one is kept) -- or, in the last Combine of a step,
// applies the parameter update to W in place of storing X.
#pragma once

#include <stdint.h>

#include "internal.h"
#include "ptx.cuh"

namespace dmuon {

// One 32-column chunk of a thread's aux row: q[0..3] the bf16 values, and
// q[4..7] their bf16 low halves when lo_row is given.
__device__ __forceinline__ void load_aux_chunk(const uint16_t* hi_row, const uint16_t* lo_row, int c0,
                                               uint4 (&q)[8]) {
  const uint4* h = reinterpret_cast<const uint4*>(hi_row + c0);
#pragma unroll
  for (int i = 0; i < 4; ++i) q[i] = __ldg(h + i);
  if (lo_row) {
    const uint4* l = reinterpret_cast<const uint4*>(lo_row + c0);
#pragma unroll
    for (int i = 0; i < 4; ++i) q[4 + i] = __ldg(l + i);
  }
}

__device__ __forceinline__ void unpack_aux_chunk(const uint4 (&q)[8], bool has_lo, float (&f)[32]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t w[4] = {q[i].x, q[i].y, q[i].z, q[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      f[8 * i + 2 * j] = __uint_as_float(w[j] << 16);
      f[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
  }
  if (has_lo) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t w[4] = {q[4 + i].x, q[4 + i].y, q[4 + i].z, q[4 + i].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        f[8 * i + 2 * j] += __uint_as_float(w[j] << 16);
        f[8 * i + 2 * j + 1] += __uint_as_float(w[j] & 0xFFFF0000u);
      }
    }
  }
}

// row_in_tile: this thread's row within the tile; tmem_lane_base: TMEM
// address of this warp's lane quarter at column 0 of the accumulator.
// Tiles are 256 columns wide; `mirror` tiles are strictly above the
// diagonal of a symmetric output.
template <bool FUSE>
__device__ __forceinline__ void ns_epilogue_tile(const NsLaunch& L, const NsProblem& P, int m0, int n0,
                                                 int row_in_tile, uint32_t tmem_lane_base, bool mirror) {
  constexpr int BN = 256;
  const uint32_t t_lane = tmem_lane_base;
  float g = 1.f;
  if (L.gscale && L.gpow > 0) {
    const float s = L.gscale[P.slice];
    g = (L.gpow == 2) ? s * s : s;
  }
  float alpha, beta;
  if (L.kind == kGram) {
    alpha = g;
    beta = 0.f;
  } else if (L.kind == kPoly) {
    alpha = L.c;
    beta = L.b;
  } else {
    alpha = g;
    beta = g * L.a;
  }
  const float diag = (L.kind == kPoly) ? L.diag : 0.f;
  const int row = m0 + row_in_tile;
  const bool row_ok = row < P.M;
  // A warp whose 32 rows all lie past the output's last row has nothing to
  // read or write (the accumulator lanes are simply left for the next tile).
  if (row - static_cast<int>(threadIdx.x & 31) >= P.M) return;
  uint16_t* out_row = reinterpret_cast<uint16_t*>(P.out) + static_cast<int64_t>(row) * P.ld_out;
  const uint16_t* aux_row =
      reinterpret_cast<const uint16_t*>(P.aux) + static_cast<int64_t>(row) * P.ld_aux;
  const uint16_t* auxlo_row = P.aux_lo ? P.aux_lo + static_cast<int64_t>(row) * P.ld_aux : nullptr;
  uint16_t* outlo_row = P.out_lo ? P.out_lo + static_cast<int64_t>(row) * P.ld_out : nullptr;
  // Fused update (last iteration): W <- W*decay - step*X, param <- bf16(W).
  constexpr bool fuse = FUSE;
  float* w_row = nullptr;
  uint16_t* p_row = nullptr;
  float decay = 1.f, step = 0.f;
  bool w_vec = false;
  if (fuse) {
    const SliceDesc& S = L.slices[P.slice];
    w_row = S.master + static_cast<int64_t>(row) * S.n;
    p_row = S.param ? S.param + static_cast<int64_t>(row) * S.n : nullptr;
    decay = 1.0f - L.lr * L.wd;
    step = L.lr * S.shape_scale;
    w_vec = S.vec_ok != 0;
  }
  // The aux operand of chunk cc+1 is loaded while chunk cc is processed, so
  // the global-load latency overlaps the TMEM read and the stores.
  const bool need_aux = beta != 0.f && row_ok;
  auto load_aux = [&](int cc, uint4 (&q)[8]) {
    const int c0 = n0 + cc * 32;
    if (!need_aux || c0 + 32 > P.N) return;
    load_aux_chunk(aux_row, auxlo_row, c0, q);
  };
  auto aux_at = [&](int c) {
    return bf16_bits_to_f32(aux_row[c]) + (auxlo_row ? bf16_bits_to_f32(auxlo_row[c]) : 0.f);
  };
  uint4 aux_next[8];
  load_aux(0, aux_next);
#pragma unroll 1
  for (int cc = 0; cc < BN / 32; ++cc) {
    const int col0 = n0 + cc * 32;
    if (col0 >= P.N) break;  // warp-uniform
    uint4 aux_cur[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) aux_cur[i] = aux_next[i];
    if (cc + 1 < BN / 32) load_aux(cc + 1, aux_next);
    __syncwarp();
    uint32_t r[32];
    tmem_ld_32x32b_x32(t_lane + static_cast<uint32_t>(cc * 32), r);
    const bool full_chunk = (col0 + 32 <= P.N);
    float auxf[32];
    if (need_aux && full_chunk) unpack_aux_chunk(aux_cur, auxlo_row != nullptr, auxf);
    float4 wq[8];
    if (fuse && row_ok && full_chunk && w_vec) {
      const float4* src = reinterpret_cast<const float4*>(w_row + col0);
#pragma unroll
      for (int i = 0; i < 8; ++i) wq[i] = src[i];
    }
    tmem_ld_wait();
    if (!row_ok) {
      // rows past M: nothing to store
    } else if (full_chunk && fuse) {
      float w[32];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (w_vec) {
          w[4 * i] = wq[i].x; w[4 * i + 1] = wq[i].y; w[4 * i + 2] = wq[i].z; w[4 * i + 3] = wq[i].w;
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k) w[4 * i + k] = w_row[col0 + 4 * i + k];
        }
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        float v = alpha * __uint_as_float(r[j]);
        if (beta != 0.f) v = fmaf(beta, auxf[j], v);
        w[j] = fmaf(-step, v, w[j] * decay);
      }
      if (w_vec) {
        float4* wd4 = reinterpret_cast<float4*>(w_row + col0);
#pragma unroll
        for (int i = 0; i < 8; ++i) wd4[i] = make_float4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        if (p_row) {
          uint4* pd = reinterpret_cast<uint4*>(p_row + col0);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            pd[i] = make_uint4(pack_bf16x2(w[8 * i], w[8 * i + 1]), pack_bf16x2(w[8 * i + 2], w[8 * i + 3]),
                               pack_bf16x2(w[8 * i + 4], w[8 * i + 5]), pack_bf16x2(w[8 * i + 6], w[8 * i + 7]));
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          w_row[col0 + j] = w[j];
          if (p_row) p_row[col0 + j] = to_bf16_bits(w[j]);
        }
      }
    } else if (full_chunk) {
      float v[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        v[j] = alpha * __uint_as_float(r[j]);
        if (beta != 0.f) v[j] = fmaf(beta, auxf[j], v[j]);
        if (row == col0 + j) v[j] += diag;
      }
      uint4* dst = reinterpret_cast<uint4*>(out_row + col0);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        dst[i] = make_uint4(pack_bf16x2(v[8 * i], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                            pack_bf16x2(v[8 * i + 4], v[8 * i + 5]), pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
      if (outlo_row) {
        uint4* dl = reinterpret_cast<uint4*>(outlo_row + col0);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          dl[i] = make_uint4(pack_bf16x2_remainder(v[8 * i], v[8 * i + 1]),
                             pack_bf16x2_remainder(v[8 * i + 2], v[8 * i + 3]),
                             pack_bf16x2_remainder(v[8 * i + 4], v[8 * i + 5]),
                             pack_bf16x2_remainder(v[8 * i + 6], v[8 * i + 7]));
      }
      if (mirror) {
        // Transposed copy: for each column j the warp's 32 lanes hold 32
        // consecutive rows, so every store instruction writes one
        // contiguous 64-byte run.
        uint16_t* mo = reinterpret_cast<uint16_t*>(P.out) + row;
#pragma unroll
        for (int j = 0; j < 32; ++j) mo[static_cast<int64_t>(col0 + j) * P.ld_out] = to_bf16_bits(v[j]);
        if (P.out_lo) {
          uint16_t* ml = P.out_lo + row;
#pragma unroll
          for (int j = 0; j < 32; ++j) ml[static_cast<int64_t>(col0 + j) * P.ld_out] = to_bf16_bits(bf16_remainder(v[j]));
        }
      }
    } else {
      for (int j = 0; j < 32 && col0 + j < P.N; ++j) {
        float v = alpha * __uint_as_float(r[j]);
        if (beta != 0.f) v = fmaf(beta, aux_at(col0 + j), v);
        if (row == col0 + j) v += diag;
        if (fuse) {
          const float w = fmaf(-step, v, w_row[col0 + j] * decay);
          w_row[col0 + j] = w;
          if (p_row) p_row[col0 + j] = to_bf16_bits(w);
          continue;
        }
        const uint16_t vb = to_bf16_bits(v);
        const uint16_t vl = to_bf16_bits(bf16_remainder(v));
        out_row[col0 + j] = vb;
        if (outlo_row) outlo_row[col0 + j] = vl;
        if (mirror) {
          const int64_t mi = static_cast<int64_t>(col0 + j);
          reinterpret_cast<uint16_t*>(P.out)[mi * P.ld_out + row] = vb;
          if (P.out_lo) P.out_lo[mi * P.ld_out + row] = vl;
        }
      }
    }
  }
}

}  // namespace dmuon

namespace dmuon {

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Epilogue of the CTA-pair kernel for a bf16 output: the warp stages each
// 32-row x 64-column box of its result in shared memory (128-byte swizzle:
// the 16-byte piece j of row r sits at r*128 + ((j ^ (r & 7)) * 16), so a
// warp's stores hit distinct banks) and lane 0 writes the box with one TMA
// tile store (asynchronous, edges clipped by the hardware).  Two 4 KiB
// buffers per warp alternate; before refilling one, lane 0 waits until the
// store issued two boxes earlier has finished reading it.  The mirrored
// copy (when symmetric outputs are not kept as upper blocks) is still
// stored directly.  The warp covers the
// 32-column chunks [c_begin, c_end) of the tile (c_begin even: whole boxes).
__device__ __forceinline__ void ns_epilogue_tile_staged(const NsLaunch& L, const NsProblem& P, int m0, int n0,
                                                        int row_in_tile, uint32_t t_lane, bool mirror,
                                                        uint32_t stage_smem, uint32_t& box_count,
                                                        int c_begin, int c_end) {
  constexpr int BN = 256;
  const int lane = threadIdx.x & 31;
  float g = 1.f;
  if (L.gscale && L.gpow > 0) {
    const float s = L.gscale[P.slice];
    g = (L.gpow == 2) ? s * s : s;
  }
  float alpha, beta;
  if (L.kind == kGram) {
    alpha = g;
    beta = 0.f;
  } else if (L.kind == kPoly) {
    alpha = L.c;
    beta = L.b;
  } else {
    alpha = g;
    beta = g * L.a;
  }
  const float diag = (L.kind == kPoly) ? L.diag : 0.f;
  const int row = m0 + row_in_tile;
  const bool row_ok = row < P.M;
  const int warp_row0 = row - lane;
  if (warp_row0 >= P.M) return;  // no row of this warp is in the output
  // The problem's width and slice coordinate, read once: every inline-asm
  // statement below clobbers memory, so a field read through P inside the
  // loop would be fetched again after each of them.
  const int PN = P.N, pz = P.z;
  const uint16_t* aux_row = reinterpret_cast<const uint16_t*>(P.aux) + static_cast<int64_t>(row) * P.ld_aux;
  const uint16_t* auxlo_row = P.aux_lo ? P.aux_lo + static_cast<int64_t>(row) * P.ld_aux : nullptr;
  const CUtensorMap* map_out = L.maps + P.map_out;
  // With a low-half output both staging buffers of the warp hold one
  // 64-column group (value and remainder), written by two TMA stores.
  const bool has_lo = P.out_lo != nullptr;
  const CUtensorMap* map_out_lo = has_lo ? L.maps + P.map_out_lo : nullptr;
  const int n_boxes = (min(BN, P.N - n0) + 63) / 64;
  const int cc_end = min(c_end, 2 * n_boxes);

  const bool need_aux = beta != 0.f && row_ok;
  auto load_aux = [&](int cc, uint4 (&q)[8]) {
    const int c0 = n0 + cc * 32;
    if (!need_aux || c0 + 32 > PN) return;
    load_aux_chunk(aux_row, auxlo_row, c0, q);
  };
  uint4 aux_next[8];
  load_aux(c_begin, aux_next);
#pragma unroll 1
  for (int cc = c_begin; cc < cc_end; ++cc) {
    const int col0 = n0 + cc * 32;
    uint4 aux_cur[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) aux_cur[i] = aux_next[i];
    if (cc + 1 < cc_end) load_aux(cc + 1, aux_next);
    __syncwarp();
    uint32_t r[32];
    tmem_ld_32x32b_x32(t_lane + static_cast<uint32_t>(cc * 32), r);
    const bool full_chunk = (col0 + 32 <= PN);
    float auxf[32];
    if (need_aux && full_chunk) {
      unpack_aux_chunk(aux_cur, auxlo_row != nullptr, auxf);
    } else if (need_aux) {
      for (int j = 0; j < 32; ++j) {
        const int c = col0 + j;
        auxf[j] = (c < PN) ? bf16_bits_to_f32(aux_row[c]) + (auxlo_row ? bf16_bits_to_f32(auxlo_row[c]) : 0.f)
                            : 0.f;
      }
    }
    tmem_ld_wait();
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      v[j] = alpha * __uint_as_float(r[j]);
      if (need_aux) v[j] = fmaf(beta, auxf[j], v[j]);
      if (row == col0 + j) v[j] += diag;
    }
    const uint32_t buf = has_lo ? stage_smem : stage_smem + (box_count & 1u) * 4096u;
    if ((cc & 1) == 0) {
      // Before refilling: the store that last read this buffer has read it
      // (with a low half both buffers are refilled, so wait for all).
      if (lane == 0) {
        if (has_lo)
          bulk_wait_group_read<0>();
        else
          bulk_wait_group_read<1>();
      }
      __syncwarp();
    }
    const uint32_t swz = static_cast<uint32_t>(lane) * 128u;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t j = static_cast<uint32_t>(4 * (cc & 1) + i);
      const uint32_t off = swz + ((j ^ static_cast<uint32_t>(lane & 7)) << 4);
      st_shared_v4(buf + off, pack_bf16x2(v[8 * i], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                   pack_bf16x2(v[8 * i + 4], v[8 * i + 5]), pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
      if (has_lo)
        st_shared_v4(buf + 4096u + off, pack_bf16x2_remainder(v[8 * i], v[8 * i + 1]),
                     pack_bf16x2_remainder(v[8 * i + 2], v[8 * i + 3]),
                     pack_bf16x2_remainder(v[8 * i + 4], v[8 * i + 5]),
                     pack_bf16x2_remainder(v[8 * i + 6], v[8 * i + 7]));
    }
    if (row_ok && mirror) {
      uint16_t* mo = reinterpret_cast<uint16_t*>(P.out) + row;
      for (int j = 0; j < 32 && col0 + j < P.N; ++j) {
        mo[static_cast<int64_t>(col0 + j) * P.ld_out] = to_bf16_bits(v[j]);
        if (has_lo) P.out_lo[static_cast<int64_t>(col0 + j) * P.ld_out + row] = to_bf16_bits(bf16_remainder(v[j]));
      }
    }
    if (cc & 1) {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_3d(map_out, buf, n0 + 64 * (cc >> 1), warp_row0, pz);
        if (has_lo) tma_store_3d(map_out_lo, buf + 4096u, n0 + 64 * (cc >> 1), warp_row0, pz);
        bulk_commit_group();
      }
      ++box_count;
    }
  }
  if (has_lo) {
    // Leave both buffers free for the next tile, whichever kind it is.
    if (lane == 0) bulk_wait_group_read<0>();
    __syncwarp();
  }
}

}  // namespace dmuon

namespace dmuon {

// The staged epilogue for launches without an aux operand (the Gram, and the
// Combine once a*X is folded into the polynomial matrix), with the TMEM
// drain software-pipelined: the load of chunk cc+1 is in flight while chunk
// cc is scaled, packed and staged, so the TMEM latency is paid once per tile
// instead of once per chunk.  Used where the epilogue is not hidden behind
// another tile's main loop: the 256 x 512 tiles (their two accumulators fill
// all of TMEM) and launches with main loops as short as the drain (8
// epilogue warps).  Same arithmetic as ns_epilogue_tile_staged with
// beta = 0, so the results are bit-identical.
__device__ __forceinline__ void ns_epilogue_tile_staged_pipe(const NsLaunch& L, const NsProblem& P, int m0, int n0,
                                                             int row_in_tile, uint32_t t_lane, uint32_t stage_smem,
                                                             uint32_t& box_count, int c_begin, int c_end) {
  constexpr int BN = 256;
  const int lane = threadIdx.x & 31;
  float alpha = 1.f;
  if (L.gscale && L.gpow > 0) {
    const float s = L.gscale[P.slice];
    alpha = (L.gpow == 2) ? s * s : s;
  }
  const float diag = (L.kind == kPoly) ? L.diag : 0.f;
  const int row = m0 + row_in_tile;
  const int warp_row0 = row - lane;
  if (warp_row0 >= P.M) return;  // no row of this warp is in the output
  const CUtensorMap* map_out = L.maps + P.map_out;
  const int pz = P.z;  // read once (the asm statements in the loop clobber memory)
  const bool has_lo = P.out_lo != nullptr;
  const CUtensorMap* map_out_lo = has_lo ? L.maps + P.map_out_lo : nullptr;
  const int n_boxes = (min(BN, P.N - n0) + 63) / 64;
  const int cc_end = min(c_end, 2 * n_boxes);
  if (c_begin >= cc_end) return;
  uint32_t nxt[32];
  __syncwarp();
  tmem_ld_32x32b_x32(t_lane + static_cast<uint32_t>(c_begin * 32), nxt);
#pragma unroll 1
  for (int cc = c_begin; cc < cc_end; ++cc) {
    const int col0 = n0 + cc * 32;
    tmem_ld_wait_regs(nxt);
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      v[j] = alpha * __uint_as_float(nxt[j]);
      if (row == col0 + j) v[j] += diag;
    }
    __syncwarp();
    if (cc + 1 < cc_end) tmem_ld_32x32b_x32(t_lane + static_cast<uint32_t>((cc + 1) * 32), nxt);
    const uint32_t buf = has_lo ? stage_smem : stage_smem + (box_count & 1u) * 4096u;
    if ((cc & 1) == 0) {
      if (lane == 0) {
        if (has_lo)
          bulk_wait_group_read<0>();
        else
          bulk_wait_group_read<1>();
      }
      __syncwarp();
    }
    const uint32_t swz = static_cast<uint32_t>(lane) * 128u;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t j = static_cast<uint32_t>(4 * (cc & 1) + i);
      const uint32_t off = swz + ((j ^ static_cast<uint32_t>(lane & 7)) << 4);
      st_shared_v4(buf + off, pack_bf16x2(v[8 * i], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                   pack_bf16x2(v[8 * i + 4], v[8 * i + 5]), pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
      if (has_lo)
        st_shared_v4(buf + 4096u + off, pack_bf16x2_remainder(v[8 * i], v[8 * i + 1]),
                     pack_bf16x2_remainder(v[8 * i + 2], v[8 * i + 3]),
                     pack_bf16x2_remainder(v[8 * i + 4], v[8 * i + 5]),
                     pack_bf16x2_remainder(v[8 * i + 6], v[8 * i + 7]));
    }
    if (cc & 1) {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_3d(map_out, buf, n0 + 64 * (cc >> 1), warp_row0, pz);
        if (has_lo) tma_store_3d(map_out_lo, buf + 4096u, n0 + 64 * (cc >> 1), warp_row0, pz);
        bulk_commit_group();
      }
      ++box_count;
    }
  }
  if (has_lo) {
    if (lane == 0) bulk_wait_group_read<0>();
    __syncwarp();
  }
}

}  // namespace dmuon

namespace dmuon {

// The last Combine's fused update on the CTA-pair kernel, with W read and
// the results written by TMA tile copies.  Per 32-column chunk a warp loads
// the 32 x 32 fp32 box of W under its rows (cp.async.bulk.tensor through the
// slice's map S.map_w in L.cmaps, 128-byte swizzle: 16-byte piece j of row r
// at r*128 + ((j ^ (r & 7)) * 16); parts past the tensor's edge read as
// zero), computes W' = W*(1 - lr*wd) - lr*scale*X in place in that box and
// the bf16 parameter into half of a 32 x 64 bf16 box, and lane 0 stores both
// boxes (rows and columns past the edge clipped by the hardware).
//
// Per warp: W boxes rotate through kFusedWBoxes 4 KiB buffers at
// stage_smem, each with its own mbarrier (wbar0 + 8*i) that the load
// completes; parameter boxes alternate between two buffers after them.  A
// warp counts the W boxes it has requested (w_issued) and consumed
// (w_used) over all its tiles: box g goes to buffer g % kFusedWBoxes and
// is the (g / kFusedWBoxes)-th completion of that buffer's barrier.
// fused_w_prefetch requests a tile's first kFusedWAhead boxes before the
// epilogue waits for the tile's accumulator (the main loop hides them) and,
// after short main loops, prefetches the others into L2; the chunk loop
// requests box cc + kFusedWAhead after storing chunk cc, once the store of
// chunk cc - 1 (the buffer's previous user) has finished reading it.
// Same arithmetic as ns_epilogue_tile<true>, so the results are
// bit-identical to it.
constexpr int kFusedWBoxes = 3;
constexpr int kFusedWAhead = kFusedWBoxes - 1;  // boxes requested ahead of the one in use

__device__ __forceinline__ void ld_shared_v4(uint32_t addr, float (&v)[4]) {
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3])
               : "r"(addr)
               : "memory");
}

struct FusedTile {
  const CUtensorMap* map_w;
  int warp_row0, z, n_chunks;
  bool any_row;  // some row of this warp lies in the output
};

__device__ __forceinline__ FusedTile fused_tile(const NsLaunch& L, const NsProblem& P, int n0, int row) {
  const int lane = threadIdx.x & 31;
  const SliceDesc& S = L.slices[P.slice];
  FusedTile f;
  f.map_w = L.cmaps + S.map_w;
  f.warp_row0 = row - lane;
  f.z = S.z_t;
  f.n_chunks = min(8, (P.N - n0 + 31) / 32);
  f.any_row = f.warp_row0 < P.M;
  return f;
}

// Lane 0 requests W box `g` (chunk cc of the tile) into its buffer.
__device__ __forceinline__ void fused_w_request(const FusedTile& f, int n0, int cc, uint32_t g, uint32_t stage_smem,
                                                uint32_t wbar0) {
  const uint32_t b = g % kFusedWBoxes;
  mbar_expect_tx(wbar0 + 8u * b, 4096u);
  tma_load_3d(stage_smem + b * 4096u, f.map_w, wbar0 + 8u * b, n0 + 32 * cc, f.warp_row0, f.z);
}

// A tile's first two W boxes, requested before its accumulator is ready.
__device__ __forceinline__ void fused_w_prefetch(const NsLaunch& L, const NsProblem& P, int m0, int n0,
                                                 int row_in_tile, uint32_t stage_smem, uint32_t wbar0,
                                                 uint32_t& w_issued) {
  const FusedTile f = fused_tile(L, P, n0, m0 + row_in_tile);
  if (!f.any_row) return;
  const int first = min(kFusedWAhead, f.n_chunks);
  if ((threadIdx.x & 31) == 0) {
    // Their buffers' previous users are boxes w_issued - kFusedWBoxes up to
    // w_issued - 2: at most the last store (box w_issued - 1) may still be
    // reading.
    bulk_wait_group_read<1>();
    for (int cc = 0; cc < first; ++cc) fused_w_request(f, n0, cc, w_issued + cc, stage_smem, wbar0);
    // Main loops of up to 32 k-blocks are shorter than the fused epilogue,
    // whose W boxes then arrive late: the tile's other W boxes are brought
    // into L2 while the main loop runs, so their loads into shared memory
    // (kFusedWAhead chunks ahead) hit L2 (GPT-2 set -1.0 %, many-small
    // -1.1 %).
    // Longer main loops hide the W loads already, and the extra requests
    // there only compete with the operand copies (Llama-3-8B +1 to +3 ms).
    if (P.K <= 32 * 64)
      for (int cc = first; cc < f.n_chunks; ++cc) tma_prefetch_l2_3d(f.map_w, n0 + 32 * cc, f.warp_row0, f.z);
  }
  w_issued += first;
}

// Returns false when a wait for a W box ran out (the block is aborting).
__device__ __forceinline__ bool ns_epilogue_tile_fused_tma(const NsLaunch& L, const NsProblem& P, int m0, int n0,
                                                           int row_in_tile, uint32_t t_lane, uint32_t stage_smem,
                                                           uint32_t wbar0, uint32_t& w_issued, uint32_t& w_used,
                                                           volatile int* abort_flag) {
  const int lane = threadIdx.x & 31;
  float g = 1.f;
  if (L.gscale && L.gpow > 0) {
    const float s = L.gscale[P.slice];
    g = (L.gpow == 2) ? s * s : s;
  }
  const float alpha = g, beta = g * L.a;
  // The problem's fields the chunk loop uses, read once: every inline-asm
  // statement below clobbers memory, so a field read through P inside the
  // loop would be fetched again after each of them.
  const int PN = P.N;
  const int row = m0 + row_in_tile;
  const bool row_ok = row < P.M;
  const FusedTile f = fused_tile(L, P, n0, row);
  if (!f.any_row) return true;  // no row of this warp is in the output
  const SliceDesc& S = L.slices[P.slice];
  const float decay = 1.0f - L.lr * L.wd;
  const float step = L.lr * S.shape_scale;
  const CUtensorMap* map_p = S.map_p >= 0 ? L.cmaps + S.map_p : nullptr;
  const uint16_t* aux_row = reinterpret_cast<const uint16_t*>(P.aux) + static_cast<int64_t>(row) * P.ld_aux;
  const uint16_t* auxlo_row = P.aux_lo ? P.aux_lo + static_cast<int64_t>(row) * P.ld_aux : nullptr;
  const bool need_aux = beta != 0.f && row_ok;
  auto load_aux = [&](int cc, uint4 (&q)[8]) {
    const int c0 = n0 + cc * 32;
    if (c0 + 32 > PN) return;
    load_aux_chunk(aux_row, auxlo_row, c0, q);
  };
  const int n_chunks = f.n_chunks;
  const uint32_t swz = static_cast<uint32_t>(lane) * 128u;
  const uint32_t pbase = stage_smem + static_cast<uint32_t>(kFusedWBoxes) * 4096u;
  uint4 aux_next[8];
  if (need_aux) load_aux(0, aux_next);
#pragma unroll 1
  for (int cc = 0; cc < n_chunks; ++cc) {
    const int col0 = n0 + cc * 32;
    uint4 aux_cur[8];
    float auxf[32];
    if (need_aux) {
#pragma unroll
      for (int i = 0; i < 8; ++i) aux_cur[i] = aux_next[i];
      if (cc + 1 < n_chunks) load_aux(cc + 1, aux_next);
    }
    __syncwarp();
    uint32_t r[32];
    tmem_ld_32x32b_x32(t_lane + static_cast<uint32_t>(cc * 32), r);
    if (need_aux) {
      if (col0 + 32 <= PN) {
        unpack_aux_chunk(aux_cur, auxlo_row != nullptr, auxf);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int c = col0 + j;
          auxf[j] = (c < PN) ? bf16_bits_to_f32(aux_row[c]) + (auxlo_row ? bf16_bits_to_f32(auxlo_row[c]) : 0.f)
                             : 0.f;
        }
      }
    }
    const uint32_t gbox = w_used + static_cast<uint32_t>(cc);
    const uint32_t wbuf = stage_smem + (gbox % kFusedWBoxes) * 4096u;
    const bool w_ready = mbar_wait_bounded(wbar0 + 8u * (gbox % kFusedWBoxes), (gbox / kFusedWBoxes) & 1u,
                                           abort_flag, L.err, kErrTimeoutEpilogue);
    tmem_ld_wait_regs(r);
    if (!w_ready) {
      w_used += static_cast<uint32_t>(cc);
      return false;
    }
    float w[32];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float q[4];
      ld_shared_v4(wbuf + swz + ((static_cast<uint32_t>(j) ^ static_cast<uint32_t>(lane & 7)) << 4), q);
      w[4 * j] = q[0]; w[4 * j + 1] = q[1]; w[4 * j + 2] = q[2]; w[4 * j + 3] = q[3];
    }
    // Rows past the output's edge (need_aux false there) are clipped by the
    // stores, so only the in-range rows' values matter.
    if (need_aux) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        w[j] = fmaf(-step, fmaf(beta, auxf[j], alpha * __uint_as_float(r[j])), w[j] * decay);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) w[j] = fmaf(-step, alpha * __uint_as_float(r[j]), w[j] * decay);
    }
    // The parameter buffer of this chunk: free once at most the previous
    // chunk's stores are still reading shared memory.
    if (lane == 0 && map_p) bulk_wait_group_read<1>();
    __syncwarp();
    const uint32_t pbuf = pbase + static_cast<uint32_t>((cc >> 1) & 1) * 4096u;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t off = swz + ((static_cast<uint32_t>(j) ^ static_cast<uint32_t>(lane & 7)) << 4);
      st_shared_v4(wbuf + off, __float_as_uint(w[4 * j]), __float_as_uint(w[4 * j + 1]),
                   __float_as_uint(w[4 * j + 2]), __float_as_uint(w[4 * j + 3]));
    }
    if (map_p) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t j = static_cast<uint32_t>(4 * (cc & 1) + i);
        const uint32_t off = swz + ((j ^ static_cast<uint32_t>(lane & 7)) << 4);
        st_shared_v4(pbuf + off, pack_bf16x2(w[8 * i], w[8 * i + 1]), pack_bf16x2(w[8 * i + 2], w[8 * i + 3]),
                     pack_bf16x2(w[8 * i + 4], w[8 * i + 5]), pack_bf16x2(w[8 * i + 6], w[8 * i + 7]));
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_3d(f.map_w, wbuf, col0, f.warp_row0, f.z);
      // A parameter box holds two chunks; the last chunk of a ragged tile
      // stores its half alone (the other half lies past the edge).
      if (map_p && ((cc & 1) || cc + 1 == n_chunks))
        tma_store_3d(map_p, pbuf, n0 + 64 * (cc >> 1), f.warp_row0, f.z);
      bulk_commit_group();
      if (cc + kFusedWAhead < n_chunks) {
        // Box cc + kFusedWAhead reuses the buffer of chunk cc - 1: wait
        // until at most this chunk's stores are still reading.
        bulk_wait_group_read<1>();
        fused_w_request(f, n0, cc + kFusedWAhead, gbox + kFusedWAhead, stage_smem, wbar0);
      }
    }
    if (cc + kFusedWAhead < n_chunks) ++w_issued;
  }
  w_used += static_cast<uint32_t>(n_chunks);
  return true;
}

}  // namespace dmuon
