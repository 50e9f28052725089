// Internal types shared by the host planner (api.cu) and the kernels.
// Not part of the public ABI (include/dmuon.h is).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dmuon {

// Device error word values (written by kernels, read by dmuon_sync).
enum : int {
  kErrNone = 0,
  kErrTimeoutProducer = 1,
  kErrTimeoutMma = 2,
  kErrTimeoutEpilogue = 3,
  kErrTimeoutDrain = 4,
  kErrTimeoutSelftest = 5,
};

// One 2-D slice (m x n, row-major, contiguous) of a Muon tensor, as the two
// streaming passes see it.  Pointers already point at the slice's first
// element.  The Newton-Schulz workspace holds the slice as m rows of `ld`
// elements (ld >= n, padded so every row starts on a 16-byte boundary).
struct SliceDesc {
  float* master;
  float* momentum;
  const void* grad;
  uint16_t* param;        // may be null
  void* x0;               // workspace: X before the first iteration (NS operand dtype)
  uint16_t* x0lo;         // workspace: low bf16 half of X0, X0 - bf16(X0) (bf16 path), or null
  const void* xk;         // workspace: X after the last iteration
  int64_t ld;             // workspace row pitch, elements
  int32_t m, n;
  int32_t grad_bf16;      // 1: grad is bf16, 0: fp32
  int32_t vec_ok;         // 1: n % 8 == 0 and every pointer 16-byte aligned
  float shape_scale;      // sqrt(max(1, m/n))
  int32_t chunk_begin;    // first chunk of this slice in the chunk table
  int32_t chunk_end;
  int32_t x_f32;          // 1: this slice's NS workspace is fp32 (fp32 CUDA-core path)
  // Fused update with TMA stores: tensor maps (in NsLaunch::cmaps) of the
  // slice's tensor's master (fp32, 32 x 32 boxes) and bf16 parameter
  // (64 x 32 boxes, -1 = no parameter), and the slice's index within its
  // tensor (the maps' third coordinate).
  int32_t map_w, map_p, z_t;
};

// A contiguous run of one slice's elements (row-major element index of the
// m x n slice).  Start is a multiple of 8.
struct Chunk {
  int32_t slice;
  int32_t count;
  int64_t start;
};

// One AdamW tensor for the element-wise kernel.
struct VecDesc {
  float* master;
  float* exp_avg;
  float* exp_avg_sq;
  const void* grad;
  uint16_t* param;
  int32_t grad_bf16;
  int32_t vec_ok;
};

// One product of a Newton-Schulz phase: D(MxN) = A_op(MxK) * B_op(KxN),
// then an epilogue that depends on the phase kind (see NsKind).
//  - Raw view (used by the fp32 CUDA-core path): A_op(i,k) = a[i*a_si + k*a_sk],
//    B_op(k,j) = b[k*b_sk + j*b_sj].
//  - Tensor-map view (used by the tcgen05 path): operand tiles are loaded with
//    TMA from maps[map_a] / maps[map_b] at slice coordinate z; bit 0 of
//    `majors` marks A_op as M-contiguous in memory, bit 1 marks B_op as
//    N-contiguous (otherwise the operand is K-contiguous).
struct NsProblem {
  const void* a;
  const void* b;
  int64_t a_si, a_sk, b_sk, b_sj;
  void* out;
  const void* aux;
  int64_t ld_out, ld_aux;
  // tcgen05 path, first iterations: low bf16 halves (v - bf16(v)) of the aux
  // operand (read, aux + aux_lo carries 16 significant bits) and of the
  // output (written), or null.  Same pitch as aux / out.
  const uint16_t* aux_lo;
  uint16_t* out_lo;
  int32_t map_out_lo;     // tensor map of out_lo with 64 x 32 boxes (CTA-pair kernel)
  int32_t M, N, K;
  int32_t slice;          // global slice index (norm table)
  int32_t map_a, map_b;
  int32_t z;
  int32_t majors;
  // 1: the output is symmetric (Gram, Poly on the tcgen05 path).  Only tiles
  // whose 256-row block is on or above the diagonal 256-column block are
  // scheduled.  The one-CTA kernel also writes the transpose of every tile
  // strictly above the diagonal; the CTA-pair kernel (NsLaunch::tri) does
  // not, and reads such outputs through `tri` instead.
  int32_t sym;
  // Bit 0 / bit 1: A_op / B_op is a symmetric p x p matrix of which only the
  // 256-blocks on or above the diagonal are stored (CTA-pair kernel).  A
  // k-block below the diagonal is loaded from the transposed stored block
  // through the M/N-contiguous map map_a_t / map_b_t.
  int32_t tri;
  int32_t map_a_t, map_b_t;
  // Tensor map of `out` with 64 x 32 boxes, for the CTA-pair kernel's staged
  // TMA stores of bf16 outputs.
  int32_t map_out;
};

// Phase kinds of one Newton-Schulz iteration.
//   kGram:    out = g^p * acc                 (A = X X^T)
//   kPoly:    out = c * acc + b * aux          (B = b A + c A A, aux = A)
//   kCombine: out = g^p * (acc + a * aux)      (X' = a X + B X, aux = X)
// g = 1/(||u||+eps) of the slice when the fold-in of the normalisation is
// active (first iteration), p = gpow; g^0 = 1.
// On the bf16 path the MMA operands are always bf16, but the first two
// iterations keep the low halves of X0, A and X1 (aux_lo / out_lo) for the
// epilogue terms b*A and a*X: those terms carry the weak directions of a
// gradient dominated by a few large singular values, and rounding them to
// bf16 before the iteration amplifies them is what costs accuracy.  A bf16
// value plus its bf16 remainder holds 16 significant bits, which is as good
// as fp32 here and costs 2 bytes per element instead of 4.
enum NsKind : int { kGram = 0, kPoly = 1, kCombine = 2 };

// CTA-pair tile lists: bit 31 of a tile's problem index marks a 256 x 512
// tile (column blocks tile_n and tile_n + 1).
constexpr uint32_t kTileWideBit = 0x80000000u, kTileProbMask = 0x7FFFFFFFu;

struct NsLaunch {
  const NsProblem* probs;
  const uint2* tiles;       // x = problem index, y = (tile_m << 16) | tile_n
  const int32_t* cta_begin; // per persistent CTA: tiles[cta_begin[i] .. cta_begin[i+1])
  const CUtensorMap* maps;  // tcgen05 path only
  const float* gscale;      // per-slice 1/(||u||+eps), or null
  int32_t gpow;
  int32_t kind;
  float a, b, c;
  int* err;
  // Last Combine of the step on the tensor-core path: instead of storing X,
  // apply W <- W*(1 - lr*wd) - lr*shape_scale*X and the bf16 copy in the
  // epilogue (slices[P.slice] gives W, the parameter and the scale; X has the
  // orientation of W, so output (row, col) is W[row][col]).
  const SliceDesc* slices;
  int32_t fuse_update;
  float lr, wd;
  // CTA-pair kernel: symmetric outputs keep only their upper blocks (no
  // mirrored stores) and symmetric operands are read through NsProblem::tri.
  int32_t tri;
  // Poly only: added to the diagonal of B, so that the Combine of the same
  // iteration computes a X + B X as (a I + B) X without reading X as aux
  // (that Combine then runs with a = 0).  0 = off.
  float diag;
  // CTA-pair kernel: 8 epilogue warps instead of 4 (not with fuse_update).
  int32_t epi8;
  // CTA-pair kernel: the tile list holds 256 x 512 tiles (kTileWideBit);
  // needs tri, excludes fuse_update.
  int32_t wide;
  // CTA-pair kernel: ring depth of the 256 x 256 tiles (4 or 5; a launch
  // with fuse_update always runs 4).
  int32_t stages;
  // Fused update: tensor maps of the callers' masters and parameters
  // (SliceDesc::map_w / map_p index them).
  const CUtensorMap* cmaps;
};

// ---- launch wrappers (each returns the cudaError_t of its launch) ----
cudaError_t launch_momentum(const SliceDesc* slices, const Chunk* chunks, int n_chunks,
                            float mu, int nesterov, int x_fp32, float* partials,
                            cudaStream_t st);
cudaError_t launch_norm(const SliceDesc* slices, int n_slices, const float* partials,
                        float* inv_norm, cudaStream_t st);
cudaError_t launch_update(const SliceDesc* slices, const Chunk* chunks, int n_chunks,
                          float lr, float wd, int x_fp32, const float* xscale,
                          cudaStream_t st);
cudaError_t launch_adamw(const VecDesc* vecs, const Chunk* chunks, int n_chunks,
                         float lr, float beta1, float beta2, float eps, float wd,
                         float bc1, float bc2_sqrt, cudaStream_t st);
cudaError_t launch_selftest_wait(int* err, long long timeout_ns, cudaStream_t st);

cudaError_t launch_ns_tc(const NsLaunch& L, int n_ctas, cudaStream_t st);
// CTA-pair variant: tiles are kTc2Tile x kTc2Tile, cta_begin is indexed by pair.
cudaError_t launch_ns_tc2(const NsLaunch& L, int n_pairs, cudaStream_t st);
int ns_tc2_max_pairs();
cudaError_t launch_ns_simt(const NsLaunch& L, int n_tiles, cudaStream_t st);

// Function attributes (e.g. the shared-memory opt-in) are per device: one
// bit per device ordinal records that a kernel's attributes are set there.
inline bool attr_needed_on_current_device(unsigned long long* mask) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev > 63) return true;
  return (__atomic_load_n(mask, __ATOMIC_ACQUIRE) & (1ull << dev)) == 0;
}
inline void attr_note_current_device(unsigned long long* mask) {
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev <= 63)
    __atomic_fetch_or(mask, 1ull << dev, __ATOMIC_ACQ_REL);
}

// Tile geometry of the two Newton-Schulz GEMM paths.
constexpr int kTcBM = 128, kTcBN = 256, kTcBK = 64;
constexpr int kTc2Tile = 256;
constexpr int kSimtBM = 64, kSimtBN = 64;
// Slices with min(m, n) below this run Newton-Schulz on the fp32 CUDA-core
// path even in bf16 mode: with so few singular values the bf16 rounding
// error does not average out (the oracle's emulation of the bf16 path
// reaches 2.3e-2 at 24 x 256), and such products are cheap in fp32.
constexpr int kFp32BelowP = 64;
constexpr int kChunkElems = 1 << 16;

}  // namespace dmuon
