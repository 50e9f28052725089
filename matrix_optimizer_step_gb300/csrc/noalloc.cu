// dmuon_muon_step_noalloc: the Muon step for callers that cannot allocate
// device memory.
//
// Some callers may not call cudaMalloc at all: code running inside a
// framework that owns every device allocation through its own pool, code
// that must not grow its footprint after start-up, or code that must not
// synchronise the device (cudaMalloc/cudaFree can).  dmuon_muon_step needs a
// context, and a context allocates its Newton-Schulz workspace and plan
// tables on first use.  This variant allocates nothing: every byte of scratch
// (the X/A/B buffers of the iteration, the norm partials, the descriptor
// tables and the TMA tensor maps) lives in one file-scope __device__ array of
// kNoAllocScratchBytes, which the CUDA runtime reserves on every device that
// loads this library and keeps until the process exits.  The host-side
// tables (tensor maps included) are built in a file-scope host buffer, so no
// heap allocation happens either.  The caller passes inputs and outputs
// exactly as for dmuon_muon_step.
//
// The kernels are the same ones dmuon_muon_step launches (momentum, norm,
// the Newton-Schulz phases, update), with the same per-shape precision
// policy: a tensor whose slices have min(m, n) >= 64 runs Newton-Schulz on
// the bf16 tensor cores (one CTA per 128 x 256 tile), a tensor with
// min(m, n) < 64, or a call with DMUON_FLAG_FP32_NS, on the fp32 CUDA-core
// kernel.  Only where the scratch lives and how tiles are spread over the
// CTAs (round robin here: for one tensor every tile of a phase has the same
// cost) differ.
//
// Scratch layout (byte offsets into the array):
//   [0, 256)        device error word (int at offset 0); bounded waits that
//                   run out record their site here.  Never cleared by a
//                   step: dmuon_muon_step_noalloc_sync reads and clears it.
//   [256, 256 + T)  tables, uploaded in one copy from the host buffer:
//                   tensor maps, slice descriptors, chunks, problems, tiles,
//                   per-CTA tile ranges
//   then            the Newton-Schulz buffers, norm partials and norms
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "../../include/dmuon.h"
#include "host_util.h"
#include "internal.h"

namespace dmuon {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // device scratch: 64 MiB
constexpr size_t kNoAllocTableBytes = size_t(1) << 20;     // host staging of the tables: 1 MiB
constexpr size_t kErrRegion = 256;                         // error word region at offset 0
constexpr int kMaxDevices = 64;
constexpr int64_t kMaxCtas = 1024;  // tile-range table bound (a GB300 has 152 SMs)

// The scratch.  In host code `g_noalloc_scratch` names a host-side stand-in,
// not a device address: its device address comes from cudaGetSymbolAddress.
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};
alignas(128) unsigned char g_host_tables[kNoAllocTableBytes];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

int fail_cuda(cudaError_t e, const char* what) {
  char buf[160];
  snprintf(buf, sizeof buf, "muon_step_noalloc: %s: %s", what, cudaGetErrorString(e));
  return set_error(DMUON_ERR_CUDA, buf);
}

size_t up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool encode(EncodeTiledFn enc, CUtensorMap* out, void* base, int64_t inner, int64_t rows,
            int64_t count, int64_t ld, uint32_t box_inner, uint32_t box_rows) {
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)count};
  cuuint64_t strides[2] = {(cuuint64_t)(ld * 2), (cuuint64_t)(rows * ld * 2)};
  cuuint32_t box[3] = {box_inner, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Device address of the scratch on the current device, looked up once per
// device with that device current.  Caller holds g_mu.
int scratch_on_current_device(uint8_t** out, int* dev_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return set_error(DMUON_ERR_UNSUPPORTED, "muon_step_noalloc: device ordinal");
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || !ptr) return fail_cuda(e, "cudaGetSymbolAddress of the static scratch");
    g_scratch_addr[dev] = ptr;
  }
  *out = static_cast<uint8_t*>(g_scratch_addr[dev]);
  if (dev_out) *dev_out = dev;
  return DMUON_OK;
}

// Tiles of one phase: `sym` phases (tensor-core Gram and Poly) schedule only
// tiles whose row block is on or above the diagonal column block, as
// dmuon_muon_step does.  One term per row of tiles.
int64_t phase_tiles(int64_t rows, int64_t cols, int64_t bm, int64_t bn, bool sym) {
  const int64_t tm = (rows + bm - 1) / bm, tn = (cols + bn - 1) / bn;
  if (!sym) return tm * tn;
  int64_t k = 0;
  for (int64_t i = 0; i < tm; ++i) k += std::max<int64_t>(0, tn - (i * bm) / bn);
  return k;
}

}  // namespace

// The scratch's error word on the current device (for the wait self-test).
int noalloc_error_word(int** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  uint8_t* base = nullptr;
  const int st = scratch_on_current_device(&base, nullptr);
  if (st != DMUON_OK) return st;
  *out = reinterpret_cast<int*>(base);
  return DMUON_OK;
}

}  // namespace dmuon

using namespace dmuon;

extern "C" int dmuon_muon_step_noalloc(const dmuon_matrix* mat, float lr, float momentum, float wd,
                                       int32_t ns_steps, float a, float b, float c, uint32_t flags,
                                       void* stream) {
  clear_error();
  if (!mat) return set_error(DMUON_ERR_INVALID_ARG, "muon_step_noalloc: null tensor");
  if (!std::isfinite(lr) || !std::isfinite(momentum) || !std::isfinite(wd) || !std::isfinite(a) ||
      !std::isfinite(b) || !std::isfinite(c))
    return set_error(DMUON_ERR_INVALID_ARG, "muon_step_noalloc: non-finite hyper-parameter");
  if (ns_steps < 0 || ns_steps > 100)
    return set_error(DMUON_ERR_INVALID_ARG, "muon_step_noalloc: ns_steps outside [0, 100]");
  if (flags & ~uint32_t(DMUON_FLAG_NESTEROV | DMUON_FLAG_FP32_NS))
    return set_error(DMUON_ERR_INVALID_ARG, "muon_step_noalloc: unknown flag bits");
  // The checks of dmuon_muon_step: rank, every dimension in [1, 2^31], at
  // most 2^40 elements, m*n < 2^31, pointers, dtype.  After them every size
  // product below stays far inside int64.
  int st = validate_matrix(*mat, 0);
  if (st != DMUON_OK) return st;
  const dmuon_matrix& M = *mat;
  int64_t S = 1;
  for (int d = 0; d < M.rank - 2; ++d) S *= M.shape[d];
  const int64_t m = M.shape[M.rank - 2], n = M.shape[M.rank - 1];
  const int64_t p = std::min(m, n), q = std::max(m, n);
  const int64_t numel = S * m * n;  // <= 2^40
  const bool f32 = (flags & DMUON_FLAG_FP32_NS) != 0 || p < kFp32BelowP;
  // Every element needs at least two X buffers plus, on the bf16 path, X's
  // low half: 6 bytes (bf16) or 8 (fp32).  Reject on that alone before any
  // finer sizing.
  if (numel > static_cast<int64_t>(kNoAllocScratchBytes / (f32 ? 8 : 6))) {
    char buf[200];
    snprintf(buf, sizeof buf,
             "muon_step_noalloc: this tensor (%lld elements) needs more than the static limit of %zu bytes of scratch",
             (long long)numel, kNoAllocScratchBytes);
    return set_error(DMUON_ERR_SHAPE, buf);
  }
  if (check_no_overlap(mat, 1, nullptr, 0) != DMUON_OK) return DMUON_ERR_INVALID_ARG;
  const bool tall = m > n;
  const int64_t es = f32 ? 4 : 2;
  const int64_t ld = static_cast<int64_t>(up(n, 8)), ldp = static_cast<int64_t>(up(p, 8));
  const int64_t chunks_per_slice = (m * n + kChunkElems - 1) / kChunkElems;
  const int64_t n_chunks = chunks_per_slice * S;

  // Tiles per slice and phase: tensor-core 128 x 256 tiles (symmetric Gram
  // and Poly on or above the diagonal), or fp32 64 x 64 tiles (all of them).
  const int64_t comb_m = tall ? q : p, comb_n = tall ? p : q;
  const int64_t bm = f32 ? kSimtBM : kTcBM, bn = f32 ? kSimtBN : kTcBN;
  if ((comb_m + bm - 1) / bm > 0xFFFF || (comb_n + bn - 1) / bn > 0xFFFF)
    return set_error(DMUON_ERR_SHAPE, "muon_step_noalloc: matrix too large for the tile index");
  const int64_t tiles_per[3] = {phase_tiles(p, p, bm, bn, !f32), phase_tiles(p, p, bm, bn, !f32),
                                phase_tiles(comb_m, comb_n, bm, bn, false)};

  // Table region (host buffer and its device copy): tensor maps (tensor-core
  // path), slices, chunks, problems, tiles, per-CTA tile ranges.
  size_t t_off = 0;
  auto ttake = [&](size_t bytes) {
    const size_t o = t_off;
    t_off = up(t_off + bytes, 256);
    return o;
  };
  const int n_maps = f32 ? 0 : 6;
  const int n_var = f32 ? 2 : 4;
  const size_t t_maps = ttake(size_t(n_maps) * sizeof(CUtensorMap));
  const size_t t_slices = ttake(size_t(S) * sizeof(SliceDesc));
  const size_t t_chunks = ttake(size_t(n_chunks) * sizeof(Chunk));
  const size_t t_probs = ttake(size_t(3) * n_var * S * sizeof(NsProblem));
  size_t t_tiles[3], t_cta[3];
  int64_t tiles_total[3];
  for (int k = 0; k < 3; ++k) {
    tiles_total[k] = tiles_per[k] * S;
    t_tiles[k] = ttake(size_t(tiles_total[k]) * sizeof(uint2));
    t_cta[k] = ttake(f32 ? 0 : size_t(std::min(tiles_total[k], kMaxCtas) + 1) * sizeof(int32_t));
  }

  // Device buffers after the error word and the tables.
  size_t off = up(kErrRegion + t_off, 1024);
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = up(off + bytes, 1024);
    return o;
  };
  size_t o_x[2];
  o_x[0] = take(size_t(S) * m * ld * es);
  o_x[1] = take(size_t(S) * m * ld * es);
  const size_t o_xl = f32 ? 0 : take(size_t(S) * m * ld * 2);
  const size_t o_a = take(size_t(S) * p * ldp * es);
  const size_t o_al = f32 ? 0 : take(size_t(S) * p * ldp * 2);
  const size_t o_b = take(size_t(S) * p * ldp * es);
  const size_t o_part = take(size_t(n_chunks) * 4);
  const size_t o_norm = take(size_t(S) * 4);
  const size_t need = off;
  if (t_off > kNoAllocTableBytes || need > kNoAllocScratchBytes) {
    char buf[220];
    snprintf(buf, sizeof buf,
             "muon_step_noalloc: this tensor needs %zu bytes of scratch (tables %zu); the static limit is "
             "%zu bytes (tables %zu)",
             need, t_off, kNoAllocScratchBytes, kNoAllocTableBytes);
    return set_error(DMUON_ERR_SHAPE, buf);
  }

  // Device checks (first CUDA calls of the entry).
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  int major = 0, sms = 0;
  e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceGetAttribute");
  if (major != 10) return set_error(DMUON_ERR_UNSUPPORTED, "muon_step_noalloc: not an sm_100-family device");
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceGetAttribute");
  if (sms < 1 || sms > kMaxCtas) return set_error(DMUON_ERR_UNSUPPORTED, "muon_step_noalloc: SM count");

  std::lock_guard<std::mutex> lock(g_mu);
  // One-time set-up per device, with that device current.
  uint8_t* base = nullptr;
  st = scratch_on_current_device(&base, nullptr);
  if (st != DMUON_OK) return st;
  static EncodeTiledFn enc = nullptr;
  if (!f32 && !enc) {
    void* fp = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fp, 12000, cudaEnableDefault, &qr) !=
            cudaSuccess ||
        qr != cudaDriverEntryPointSuccess)
      return set_error(DMUON_ERR_CUDA, "muon_step_noalloc: cuTensorMapEncodeTiled unavailable");
    enc = reinterpret_cast<EncodeTiledFn>(fp);
  }
  uint8_t* host = g_host_tables;
  uint8_t* dtab = base + kErrRegion;

  // Tensor maps (tensor-core path): X0/X1 K-major and MN-major, A, B.
  if (!f32) {
    CUtensorMap* maps = reinterpret_cast<CUtensorMap*>(host + t_maps);
    const bool ok = encode(enc, &maps[0], base + o_x[0], n, m, S, ld, 64, 128) &&
                    encode(enc, &maps[1], base + o_x[1], n, m, S, ld, 64, 128) &&
                    encode(enc, &maps[2], base + o_x[0], n, m, S, ld, 64, 64) &&
                    encode(enc, &maps[3], base + o_x[1], n, m, S, ld, 64, 64) &&
                    encode(enc, &maps[4], base + o_a, p, p, S, ldp, 64, 128) &&
                    encode(enc, &maps[5], base + o_b, p, p, S, ldp, 64, 128);
    if (!ok) return set_error(DMUON_ERR_CUDA, "muon_step_noalloc: cuTensorMapEncodeTiled failed");
  }

  // Slices and chunks.
  SliceDesc* hs = reinterpret_cast<SliceDesc*>(host + t_slices);
  Chunk* hc = reinterpret_cast<Chunk*>(host + t_chunks);
  const bool gbf = M.grad_dtype == DMUON_DTYPE_BF16;
  for (int64_t s = 0; s < S; ++s) {
    SliceDesc D;
    memset(&D, 0, sizeof D);
    const int64_t eo = s * m * n;
    D.master = M.master + eo;
    D.momentum = M.momentum + eo;
    D.grad = static_cast<const uint8_t*>(M.grad) + eo * (gbf ? 2 : 4);
    D.param = M.param_bf16 ? M.param_bf16 + eo : nullptr;
    D.x0 = base + o_x[0] + size_t(s) * m * ld * es;
    D.x0lo = f32 ? nullptr : reinterpret_cast<uint16_t*>(base + o_xl) + size_t(s) * m * ld;
    D.x_f32 = f32 ? 1 : 0;
    D.xk = base + o_x[ns_steps & 1] + size_t(s) * m * ld * es;
    D.ld = ld;
    D.m = static_cast<int32_t>(m);
    D.n = static_cast<int32_t>(n);
    D.grad_bf16 = gbf;
    auto al = [](const void* q16) { return (reinterpret_cast<uintptr_t>(q16) & 15u) == 0; };
    D.vec_ok = (n % 8 == 0) && al(D.master) && al(D.momentum) && al(D.grad) && (!D.param || al(D.param));
    D.shape_scale = static_cast<float>(std::sqrt(std::max(1.0, double(m) / double(n))));
    D.chunk_begin = static_cast<int32_t>(s * chunks_per_slice);
    D.chunk_end = static_cast<int32_t>((s + 1) * chunks_per_slice);
    memcpy(&hs[s], &D, sizeof D);
    for (int64_t k = 0; k < chunks_per_slice; ++k) {
      Chunk ch;
      ch.slice = static_cast<int32_t>(s);
      ch.start = k * kChunkElems;
      ch.count = static_cast<int32_t>(std::min<int64_t>(kChunkElems, m * n - ch.start));
      memcpy(&hc[s * chunks_per_slice + k], &ch, sizeof ch);
    }
  }

  // Problems: [kind][variant][slice].  Tensor-core variants as in
  // dmuon_muon_step (0/1: X in buffer 0/1; 2/3: the first two iterations
  // with the low halves); fp32 variants 0/1 with the raw strided view.
  NsProblem* hp = reinterpret_cast<NsProblem*>(host + t_probs);
  const CUtensorMap* dmaps = reinterpret_cast<const CUtensorMap*>(dtab + t_maps);
  for (int64_t s = 0; s < S; ++s) {
    uint8_t* A = base + o_a + size_t(s) * p * ldp * es;
    uint8_t* Bm = base + o_b + size_t(s) * p * ldp * es;
    uint16_t* Al = f32 ? nullptr : reinterpret_cast<uint16_t*>(base + o_al) + size_t(s) * p * ldp;
    uint16_t* Xl = f32 ? nullptr : reinterpret_cast<uint16_t*>(base + o_xl) + size_t(s) * m * ld;
    for (int par = 0; par < 2; ++par) {
      uint8_t* X = base + o_x[par] + size_t(s) * m * ld * es;
      uint8_t* Xn = base + o_x[par ^ 1] + size_t(s) * m * ld * es;
      NsProblem g, y, cc;
      memset(&g, 0, sizeof g);
      memset(&y, 0, sizeof y);
      memset(&cc, 0, sizeof cc);
      g.slice = y.slice = cc.slice = static_cast<int32_t>(s);
      g.z = y.z = cc.z = static_cast<int32_t>(s);
      // Gram: A = X X^T (wide) or X^T X (tall), p x p, K = q.
      g.M = g.N = static_cast<int32_t>(p);
      g.K = static_cast<int32_t>(q);
      g.a = g.b = X;
      g.out = A;
      g.ld_out = ldp;
      if (!tall) {
        g.a_si = ld; g.a_sk = 1; g.b_sk = 1; g.b_sj = ld;
      } else {
        g.a_si = 1; g.a_sk = ld; g.b_sk = ld; g.b_sj = 1;
      }
      g.map_a = g.map_b = tall ? 2 + par : par;
      g.majors = tall ? 3 : 0;
      g.sym = f32 ? 0 : 1;
      // Poly: B = b A + c A A.
      y.M = y.N = y.K = static_cast<int32_t>(p);
      y.a = y.b = A;
      y.a_si = ldp; y.a_sk = 1; y.b_sk = ldp; y.b_sj = 1;
      y.map_a = y.map_b = 4;
      y.out = Bm;
      y.ld_out = ldp;
      y.aux = A;
      y.ld_aux = ldp;
      y.sym = f32 ? 0 : 1;
      // Combine: X' = a X + B X (wide) or a X + X B (tall).
      cc.out = Xn;
      cc.ld_out = ld;
      cc.aux = X;
      cc.ld_aux = ld;
      if (!tall) {
        cc.M = static_cast<int32_t>(p); cc.N = static_cast<int32_t>(q); cc.K = static_cast<int32_t>(p);
        cc.a = Bm; cc.a_si = ldp; cc.a_sk = 1;
        cc.b = X; cc.b_sk = ld; cc.b_sj = 1;
        cc.map_a = 5;
        cc.map_b = 2 + par;
        cc.majors = 2;
      } else {
        cc.M = static_cast<int32_t>(q); cc.N = static_cast<int32_t>(p); cc.K = static_cast<int32_t>(p);
        cc.a = X; cc.a_si = ld; cc.a_sk = 1;
        cc.b = Bm; cc.b_sk = ldp; cc.b_sj = 1;
        cc.map_a = par;
        cc.map_b = 5;
        cc.majors = 0;
      }
      NsProblem* v[3] = {&g, &y, &cc};
      for (int k = 0; k < 3; ++k) memcpy(&hp[(size_t(k) * n_var + par) * S + s], v[k], sizeof(NsProblem));
      if (f32) continue;
      if (par == 0) {
        g.out_lo = Al;
        y.aux_lo = Al;
        cc.aux_lo = Xl;
        cc.out_lo = Xl;  // X1's low half over X0's: each element is read before it is written
      } else {
        cc.aux_lo = Xl;
      }
      for (int k = 0; k < 3; ++k) memcpy(&hp[(size_t(k) * n_var + 2 + par) * S + s], v[k], sizeof(NsProblem));
    }
  }

  // Tiles.  Tensor-core path: round robin over R persistent CTAs, stored
  // CTA by CTA (tile t of the enumeration goes to CTA t mod R, position
  // t div R in its range).  fp32 path: one block per tile, in enumeration
  // order.
  int64_t ctas[3];
  for (int k = 0; k < 3; ++k) {
    const int64_t Mr = (k == 2) ? comb_m : p, Nc = (k == 2) ? comb_n : p;
    const bool sym = !f32 && k != 2;
    const int64_t tm = (Mr + bm - 1) / bm, tn = (Nc + bn - 1) / bn;
    uint2* ht = reinterpret_cast<uint2*>(host + t_tiles[k]);
    const int64_t T = tiles_total[k];
    const int64_t R = f32 ? 1 : std::max<int64_t>(1, std::min<int64_t>(sms, T));
    ctas[k] = R;
    if (!f32) {
      int32_t* hb = reinterpret_cast<int32_t*>(host + t_cta[k]);
      int64_t w = 0;
      for (int64_t r = 0; r <= R; ++r) {
        hb[r] = static_cast<int32_t>(w);
        if (r < R) w += T / R + (r < T % R ? 1 : 0);
      }
    }
    int64_t t = 0;
    for (int64_t s = 0; s < S; ++s)
      for (int64_t i = 0; i < tm; ++i)
        for (int64_t j = sym ? (i * bm) / bn : 0; j < tn; ++j) {
          uint2 u;
          u.x = static_cast<uint32_t>(s);
          u.y = (static_cast<uint32_t>(i) << 16) | static_cast<uint32_t>(j);
          const int64_t pos = f32 ? t : reinterpret_cast<int32_t*>(host + t_cta[k])[t % R] + t / R;
          memcpy(&ht[pos], &u, sizeof u);
          ++t;
        }
    if (t != T) return set_error(DMUON_ERR_INVALID_ARG, "muon_step_noalloc: tile bookkeeping");
  }

  // One upload of the tables (from the static host buffer; the copy from
  // pageable memory returns once the buffer has been consumed).
  cudaStream_t stm = static_cast<cudaStream_t>(stream);
  if ((e = cudaMemcpyAsync(dtab, host, t_off, cudaMemcpyHostToDevice, stm)) != cudaSuccess)
    return fail_cuda(e, "cudaMemcpyAsync (tables)");

  int* derr = reinterpret_cast<int*>(base);
  const SliceDesc* d_slices = reinterpret_cast<const SliceDesc*>(dtab + t_slices);
  const Chunk* d_chunks = reinterpret_cast<const Chunk*>(dtab + t_chunks);
  float* partials = reinterpret_cast<float*>(base + o_part);
  float* inv_norm = reinterpret_cast<float*>(base + o_norm);
  const int nesterov = (flags & DMUON_FLAG_NESTEROV) ? 1 : 0;
  if ((e = launch_momentum(d_slices, d_chunks, static_cast<int>(n_chunks), momentum, nesterov, 0, partials, stm)) !=
      cudaSuccess)
    return fail_cuda(e, "momentum launch");
  if ((e = launch_norm(d_slices, static_cast<int>(S), partials, inv_norm, stm)) != cudaSuccess)
    return fail_cuda(e, "norm launch");
  for (int it = 0; it < ns_steps; ++it) {
    const int variant = f32 ? (it & 1) : (it < 2 ? 2 + it : (it & 1));
    for (int kind = kGram; kind <= kCombine; ++kind) {
      NsLaunch L;
      memset(&L, 0, sizeof L);
      L.probs = reinterpret_cast<const NsProblem*>(dtab + t_probs) + (size_t(kind) * n_var + variant) * S;
      L.tiles = reinterpret_cast<const uint2*>(dtab + t_tiles[kind]);
      L.cta_begin = f32 ? nullptr : reinterpret_cast<const int32_t*>(dtab + t_cta[kind]);
      L.maps = f32 ? nullptr : dmaps;
      L.gscale = (it == 0 && kind != kPoly) ? inv_norm : nullptr;
      L.gpow = (kind == kGram) ? 2 : 1;
      L.kind = kind;
      L.a = a;
      L.b = b;
      L.c = c;
      L.err = derr;
      e = f32 ? launch_ns_simt(L, static_cast<int>(tiles_total[kind]), stm)
              : launch_ns_tc(L, static_cast<int>(ctas[kind]), stm);
      if (e != cudaSuccess) return fail_cuda(e, "NS launch");
    }
  }
  if ((e = launch_update(d_slices, d_chunks, static_cast<int>(n_chunks), lr, wd, 0,
                         ns_steps == 0 ? inv_norm : nullptr, stm)) != cudaSuccess)
    return fail_cuda(e, "update launch");
  return DMUON_OK;
}

extern "C" int dmuon_muon_step_noalloc_sync(void* stream) {
  clear_error();
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "cudaStreamSynchronize");
  std::lock_guard<std::mutex> lock(g_mu);
  uint8_t* base = nullptr;
  int dev = 0;
  int st = scratch_on_current_device(&base, &dev);
  if (st != DMUON_OK) return st;
  int word = 0;
  e = cudaMemcpyFromSymbol(&word, g_noalloc_scratch, sizeof word, 0, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail_cuda(e, "cudaMemcpyFromSymbol (error word)");
  if (word == kErrNone) return DMUON_OK;
  const int zero = 0;
  e = cudaMemcpyToSymbol(g_noalloc_scratch, &zero, sizeof zero, 0, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return fail_cuda(e, "cudaMemcpyToSymbol (error word)");
  char buf[120];
  snprintf(buf, sizeof buf, "muon_step_noalloc: a bounded device-side wait ran out (site %d) on device %d", word, dev);
  return set_error(DMUON_ERR_TIMEOUT, buf);
}
