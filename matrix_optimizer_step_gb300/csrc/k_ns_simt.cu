// fp32 Newton-Schulz phase GEMM on CUDA cores: the validation datapath.
//
// Same three phases and epilogues as the tcgen05 path (see NsKind), but with
// fp32 operands, fp32 products and fp32 storage throughout, so the result
// can be held to a 1e-4 relative error against the float64 oracle.  One
// block computes one 64x64 output tile of one problem; operands are read
// through the generic strided view of NsProblem, so the same kernel serves
// X X^T, A A and B X (or X B) in either orientation.
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace dmuon {
namespace {

constexpr int BM = kSimtBM, BN = kSimtBN, BK = 16;
constexpr int kThreads = 256;  // 16 x 16 threads, 4 x 4 outputs each

__global__ void __launch_bounds__(kThreads) ns_simt_kernel(NsLaunch L) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  const uint2 tile = L.tiles[blockIdx.x];
  const NsProblem P = L.probs[tile.x];
  const int m0 = static_cast<int>(tile.y >> 16) * BM;
  const int n0 = static_cast<int>(tile.y & 0xFFFFu) * BN;
  const float* A = reinterpret_cast<const float*>(P.a);
  const float* B = reinterpret_cast<const float*>(P.b);
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;

  float acc[4][4] = {};
  for (int k0 = 0; k0 < P.K; k0 += BK) {
    // Each thread stages 4 elements of each operand tile.
    for (int idx = threadIdx.x; idx < BM * BK; idx += kThreads) {
      const int i = idx / BK, k = idx % BK;
      const int gi = m0 + i, gk = k0 + k;
      As[k][i] = (gi < P.M && gk < P.K) ? A[gi * P.a_si + gk * P.a_sk] : 0.f;
    }
    for (int idx = threadIdx.x; idx < BN * BK; idx += kThreads) {
      const int j = idx % BN, k = idx / BN;
      const int gj = n0 + j, gk = k0 + k;
      Bs[k][j] = (gj < P.N && gk < P.K) ? B[gk * P.b_sk + gj * P.b_sj] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < BK; ++k) {
      float av[4], bv[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) av[r] = As[k][ty * 4 + r];
#pragma unroll
      for (int s = 0; s < 4; ++s) bv[s] = Bs[k][tx * 4 + s];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int s = 0; s < 4; ++s) acc[r][s] = fmaf(av[r], bv[s], acc[r][s]);
    }
    __syncthreads();
  }

  float g = 1.f;
  if (L.gscale && L.gpow > 0) {
    const float s = L.gscale[P.slice];
    g = (L.gpow == 2) ? s * s : s;
  }
  float* out = reinterpret_cast<float*>(P.out);
  const float* aux = reinterpret_cast<const float*>(P.aux);
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int i = m0 + ty * 4 + r;
    if (i >= P.M) continue;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int j = n0 + tx * 4 + s;
      if (j >= P.N) continue;
      float v = acc[r][s];
      if (L.kind == kGram) {
        v = g * v;
      } else if (L.kind == kPoly) {
        v = fmaf(L.c, v, L.b * aux[i * P.ld_aux + j]);
      } else {
        v = g * fmaf(L.a, aux[i * P.ld_aux + j], v);
      }
      out[i * P.ld_out + j] = v;
    }
  }
}

}  // namespace

cudaError_t launch_ns_simt(const NsLaunch& L, int n_tiles, cudaStream_t st) {
  if (n_tiles <= 0) return cudaSuccess;
  ns_simt_kernel<<<n_tiles, kThreads, 0, st>>>(L);
  return cudaGetLastError();
}

}  // namespace dmuon
