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
// tables are built in a file-scope host buffer, so no heap allocation happens
// either.  The caller passes inputs and outputs exactly as for
// dmuon_muon_step.
//
// The kernels are the same ones dmuon_muon_step launches (momentum, norm,
// the tcgen05 Newton-Schulz phases, update); only where their scratch lives
// and how tiles are spread over the CTAs (round robin here: for one tensor
// every tile of a phase has the same cost) differ.
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
constexpr size_t kNoAllocTableBytes = size_t(1) << 20;     // host staging of the tables
constexpr int kMaxDevices = 64;

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

}  // namespace
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
  if (flags & ~uint32_t(DMUON_FLAG_NESTEROV))
    return set_error(DMUON_ERR_INVALID_ARG,
                     "muon_step_noalloc: only DMUON_FLAG_NESTEROV is accepted (bf16 tensor-core path)");
  const dmuon_matrix& M = *mat;
  if (M.rank < 2) return set_error(DMUON_ERR_RANK_LT2, "muon_step_noalloc: rank < 2 (route it to AdamW)");
  if (M.rank > 4) return set_error(DMUON_ERR_SHAPE, "muon_step_noalloc: rank > 4");
  int64_t slices = 1;
  for (int d = 0; d < M.rank; ++d) {
    if (M.shape[d] < 1 || M.shape[d] > (int64_t(1) << 31))
      return set_error(DMUON_ERR_SHAPE, "muon_step_noalloc: dimension out of range");
    if (d < M.rank - 2) slices *= M.shape[d];
  }
  if (!M.master || !M.momentum || !M.grad)
    return set_error(DMUON_ERR_INVALID_ARG, "muon_step_noalloc: null master, momentum or grad");
  if (M.grad_dtype != DMUON_DTYPE_F32 && M.grad_dtype != DMUON_DTYPE_BF16)
    return set_error(DMUON_ERR_DTYPE, "muon_step_noalloc: grad dtype");
  if (check_no_overlap(mat, 1, nullptr, 0) != DMUON_OK) return DMUON_ERR_INVALID_ARG;
  const int64_t m = M.shape[M.rank - 2], n = M.shape[M.rank - 1];
  const int64_t p = std::min(m, n), q = std::max(m, n);
  const bool tall = m > n;
  const int64_t ld = up(n, 8), ldp = up(p, 8);
  const int64_t S = slices;

  // Scratch layout: tensor maps, then X0/X1 bf16, X low halves bf16, A bf16,
  // A low halves bf16, B bf16, chunk partials, per-slice norms, error word,
  // tables.
  const int64_t chunks_per_slice = (m * n + kChunkElems - 1) / kChunkElems;
  const int64_t n_chunks = chunks_per_slice * S;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = up(off + bytes, 1024);
    return o;
  };
  const size_t o_maps = take(6 * sizeof(CUtensorMap));
  size_t o_x[2];
  o_x[0] = take(size_t(S) * m * ld * 2);
  o_x[1] = take(size_t(S) * m * ld * 2);
  const size_t o_xl = take(size_t(S) * m * ld * 2);
  const size_t o_a = take(size_t(S) * p * ldp * 2);
  const size_t o_al = take(size_t(S) * p * ldp * 2);
  const size_t o_b = take(size_t(S) * p * ldp * 2);
  const size_t o_part = take(size_t(n_chunks) * 4);
  const size_t o_norm = take(size_t(S) * 4);
  const size_t o_err = take(16);
  const size_t o_tab = off;

  // Host tables: slices, chunks, problems (3 kinds x 4 variants x S), tiles,
  // CTA ranges.  Tile counts per phase (symmetric phases skip tiles below
  // the diagonal, as in dmuon_muon_step).
  auto count_tiles = [&](int64_t Mr, int64_t Nc, bool sym) {
    const int64_t tm = (Mr + kTcBM - 1) / kTcBM, tn = (Nc + kTcBN - 1) / kTcBN;
    int64_t k = 0;
    for (int64_t i = 0; i < tm; ++i)
      for (int64_t j = 0; j < tn; ++j)
        if (!(sym && (i * kTcBM) / kTcBN > j)) ++k;
    return k;
  };
  const int64_t comb_m = tall ? q : p, comb_n = tall ? p : q;
  const int64_t tiles_per[3] = {count_tiles(p, p, true), count_tiles(p, p, true),
                                count_tiles(comb_m, comb_n, false)};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return set_error(DMUON_ERR_UNSUPPORTED, "muon_step_noalloc: device ordinal");
  int major = 0, sms = 0;
  e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceGetAttribute");
  if (major != 10) return set_error(DMUON_ERR_UNSUPPORTED, "muon_step_noalloc: not an sm_100-family device");
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceGetAttribute");

  size_t t_off = 0;
  auto ttake = [&](size_t bytes) {
    const size_t o = t_off;
    t_off = up(t_off + bytes, 256);
    return o;
  };
  const size_t t_slices = ttake(size_t(S) * sizeof(SliceDesc));
  const size_t t_chunks = ttake(size_t(n_chunks) * sizeof(Chunk));
  const size_t t_probs = ttake(size_t(12) * S * sizeof(NsProblem));
  size_t t_tiles[3], t_cta[3];
  int64_t tiles_total[3], ctas[3];
  for (int k = 0; k < 3; ++k) {
    tiles_total[k] = tiles_per[k] * S;
    ctas[k] = std::max<int64_t>(1, std::min<int64_t>(sms, tiles_total[k]));
    t_tiles[k] = ttake(size_t(tiles_total[k]) * sizeof(uint2));
    t_cta[k] = ttake(size_t(ctas[k] + 1) * sizeof(int32_t));
  }
  const size_t need = o_tab + t_off;
  if (t_off > kNoAllocTableBytes || need > kNoAllocScratchBytes) {
    char buf[200];
    snprintf(buf, sizeof buf,
             "muon_step_noalloc: this tensor needs %zu bytes of scratch (tables %zu); the static limit is "
             "%zu bytes (tables %zu)",
             need, t_off, kNoAllocScratchBytes, kNoAllocTableBytes);
    return set_error(DMUON_ERR_SHAPE, buf);
  }

  std::lock_guard<std::mutex> lock(g_mu);
  // One-time set-up per device, with that device current.
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || !ptr) return fail_cuda(e, "cudaGetSymbolAddress of the static scratch");
    g_scratch_addr[dev] = ptr;
  }
  static EncodeTiledFn enc = nullptr;
  if (!enc) {
    void* fp = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fp, 12000, cudaEnableDefault, &qr) !=
            cudaSuccess ||
        qr != cudaDriverEntryPointSuccess)
      return set_error(DMUON_ERR_CUDA, "muon_step_noalloc: cuTensorMapEncodeTiled unavailable");
    enc = reinterpret_cast<EncodeTiledFn>(fp);
  }
  uint8_t* base = static_cast<uint8_t*>(g_scratch_addr[dev]);
  uint8_t* host = g_host_tables;
  uint8_t* dtab = base + o_tab;

  // Tensor maps: X0/X1 K-major and MN-major, A, B.
  CUtensorMap maps[6];
  bool ok = encode(enc, &maps[0], base + o_x[0], n, m, S, ld, 64, 128) &&
            encode(enc, &maps[1], base + o_x[1], n, m, S, ld, 64, 128) &&
            encode(enc, &maps[2], base + o_x[0], n, m, S, ld, 64, 64) &&
            encode(enc, &maps[3], base + o_x[1], n, m, S, ld, 64, 64) &&
            encode(enc, &maps[4], base + o_a, p, p, S, ldp, 64, 128) &&
            encode(enc, &maps[5], base + o_b, p, p, S, ldp, 64, 128);
  if (!ok) return set_error(DMUON_ERR_CUDA, "muon_step_noalloc: cuTensorMapEncodeTiled failed");

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
    D.x0 = base + o_x[0] + size_t(s) * m * ld * 2;
    D.x0lo = reinterpret_cast<uint16_t*>(base + o_xl) + size_t(s) * m * ld;
    D.xk = base + o_x[ns_steps & 1] + size_t(s) * m * ld * 2;
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

  // Problems: [kind][variant][slice]; variants as in dmuon_muon_step.
  NsProblem* hp = reinterpret_cast<NsProblem*>(host + t_probs);
  const CUtensorMap* dmaps = reinterpret_cast<const CUtensorMap*>(base + o_maps);
  for (int64_t s = 0; s < S; ++s) {
    uint8_t* A = base + o_a + size_t(s) * p * ldp * 2;
    uint8_t* Bm = base + o_b + size_t(s) * p * ldp * 2;
    uint16_t* Al = reinterpret_cast<uint16_t*>(base + o_al) + size_t(s) * p * ldp;
    uint16_t* Xl = reinterpret_cast<uint16_t*>(base + o_xl) + size_t(s) * m * ld;
    for (int par = 0; par < 2; ++par) {
      uint8_t* X = base + o_x[par] + size_t(s) * m * ld * 2;
      uint8_t* Xn = base + o_x[par ^ 1] + size_t(s) * m * ld * 2;
      NsProblem g, y, cc;
      memset(&g, 0, sizeof g);
      memset(&y, 0, sizeof y);
      memset(&cc, 0, sizeof cc);
      g.slice = y.slice = cc.slice = static_cast<int32_t>(s);
      g.z = y.z = cc.z = static_cast<int32_t>(s);
      g.M = g.N = static_cast<int32_t>(p);
      g.K = static_cast<int32_t>(q);
      g.out = A;
      g.ld_out = ldp;
      g.map_a = g.map_b = tall ? 2 + par : par;
      g.majors = tall ? 3 : 0;
      g.sym = 1;
      y.M = y.N = y.K = static_cast<int32_t>(p);
      y.map_a = y.map_b = 4;
      y.out = Bm;
      y.ld_out = ldp;
      y.aux = A;
      y.ld_aux = ldp;
      y.sym = 1;
      cc.out = Xn;
      cc.ld_out = ld;
      cc.aux = X;
      cc.ld_aux = ld;
      if (!tall) {
        cc.M = static_cast<int32_t>(p); cc.N = static_cast<int32_t>(q); cc.K = static_cast<int32_t>(p);
        cc.map_a = 5;
        cc.map_b = 2 + par;
        cc.majors = 2;
      } else {
        cc.M = static_cast<int32_t>(q); cc.N = static_cast<int32_t>(p); cc.K = static_cast<int32_t>(p);
        cc.map_a = par;
        cc.map_b = 5;
        cc.majors = 0;
      }
      NsProblem* v[3] = {&g, &y, &cc};
      for (int k = 0; k < 3; ++k) memcpy(&hp[(size_t(k) * 4 + par) * S + s], v[k], sizeof(NsProblem));
      if (par == 0) {
        g.out_lo = Al;
        y.aux_lo = Al;
        cc.aux_lo = Xl;
        cc.out_lo = Xl;
      } else {
        cc.aux_lo = Xl;
      }
      for (int k = 0; k < 3; ++k) memcpy(&hp[(size_t(k) * 4 + 2 + par) * S + s], v[k], sizeof(NsProblem));
    }
  }

  // Tiles, round robin over the CTAs, stored CTA by CTA.
  for (int k = 0; k < 3; ++k) {
    const int64_t Mr = (k == 2) ? comb_m : p, Nc = (k == 2) ? comb_n : p;
    const bool sym = k != 2;
    const int64_t tm = (Mr + kTcBM - 1) / kTcBM, tn = (Nc + kTcBN - 1) / kTcBN;
    uint2* ht = reinterpret_cast<uint2*>(host + t_tiles[k]);
    int32_t* hb = reinterpret_cast<int32_t*>(host + t_cta[k]);
    const int64_t R = ctas[k], T = tiles_total[k];
    int64_t w = 0;
    for (int64_t r = 0; r < R; ++r) {
      hb[r] = static_cast<int32_t>(w);
      int64_t t = 0;  // running index over (slice, i, j) in enumeration order
      for (int64_t s = 0; s < S; ++s)
        for (int64_t i = 0; i < tm; ++i)
          for (int64_t j = 0; j < tn; ++j) {
            if (sym && (i * kTcBM) / kTcBN > j) continue;
            if (t % R == r) {
              uint2 u;
              u.x = static_cast<uint32_t>(s);
              u.y = (static_cast<uint32_t>(i) << 16) | static_cast<uint32_t>(j);
              memcpy(&ht[w++], &u, sizeof u);
            }
            ++t;
          }
    }
    hb[R] = static_cast<int32_t>(w);
    if (w != T) return set_error(DMUON_ERR_INVALID_ARG, "muon_step_noalloc: tile bookkeeping");
  }

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* derr = reinterpret_cast<int*>(base + o_err);
  // Clear what must start at zero (the device error word), then upload the
  // tables and tensor maps.  The copies are from pageable host memory, so
  // they return once the host buffers have been consumed.
  if ((e = cudaMemsetAsync(derr, 0, 16, st)) != cudaSuccess) return fail_cuda(e, "cudaMemsetAsync");
  if ((e = cudaMemcpyAsync(base + o_maps, maps, sizeof maps, cudaMemcpyHostToDevice, st)) != cudaSuccess)
    return fail_cuda(e, "cudaMemcpyAsync (tensor maps)");
  if ((e = cudaMemcpyAsync(dtab, host, t_off, cudaMemcpyHostToDevice, st)) != cudaSuccess)
    return fail_cuda(e, "cudaMemcpyAsync (tables)");

  const SliceDesc* d_slices = reinterpret_cast<const SliceDesc*>(dtab + t_slices);
  const Chunk* d_chunks = reinterpret_cast<const Chunk*>(dtab + t_chunks);
  float* partials = reinterpret_cast<float*>(base + o_part);
  float* inv_norm = reinterpret_cast<float*>(base + o_norm);
  const int nesterov = (flags & DMUON_FLAG_NESTEROV) ? 1 : 0;
  if ((e = launch_momentum(d_slices, d_chunks, static_cast<int>(n_chunks), momentum, nesterov, 0, partials, st)) !=
      cudaSuccess)
    return fail_cuda(e, "momentum launch");
  if ((e = launch_norm(d_slices, static_cast<int>(S), partials, inv_norm, st)) != cudaSuccess)
    return fail_cuda(e, "norm launch");
  for (int it = 0; it < ns_steps; ++it) {
    const int variant = it < 2 ? 2 + it : (it & 1);
    for (int kind = kGram; kind <= kCombine; ++kind) {
      NsLaunch L;
      memset(&L, 0, sizeof L);
      L.probs = reinterpret_cast<const NsProblem*>(dtab + t_probs) + (size_t(kind) * 4 + variant) * S;
      L.tiles = reinterpret_cast<const uint2*>(dtab + t_tiles[kind]);
      L.cta_begin = reinterpret_cast<const int32_t*>(dtab + t_cta[kind]);
      L.maps = dmaps;
      L.gscale = (it == 0 && kind != kPoly) ? inv_norm : nullptr;
      L.gpow = (kind == kGram) ? 2 : 1;
      L.kind = kind;
      L.a = a;
      L.b = b;
      L.c = c;
      L.err = derr;
      if ((e = launch_ns_tc(L, static_cast<int>(ctas[kind]), st)) != cudaSuccess) return fail_cuda(e, "NS launch");
    }
  }
  if ((e = launch_update(d_slices, d_chunks, static_cast<int>(n_chunks), lr, wd, 0,
                         ns_steps == 0 ? inv_norm : nullptr, st)) != cudaSuccess)
    return fail_cuda(e, "update launch");
  return DMUON_OK;
}
