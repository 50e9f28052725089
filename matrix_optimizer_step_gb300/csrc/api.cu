// C ABI of the owner-side Muon / AdamW step: validation, planning, workspace
// and launch sequencing.  Every arithmetic step runs in the kernels of
// k_stream.cu, k_ns_tc.cu and k_ns_simt.cu; this file only decides what runs
// where.
//
// Plan (cached per shape set, rebuilt when the shapes or the precision mode
// change):
//  * every tensor of rank >= 2 is split into its 2-D slices (MindSpore
//    hyper-parallel "分布式 Muon 优化器 — 参数分组设计文档（v2）" §2.2: the last
//    two dims); slices of one shape form a class whose Newton-Schulz
//    workspace is a contiguous [count, rows, ld] array, so one 3-D TMA
//    tensor map covers the whole class;
//  * X keeps the orientation of the gradient.  For m <= n the Gram matrix is
//    X X^T and the last product B X; for m > n it is X^T X and X B.  The
//    two forms are the same iteration (transpose equivariance), and no
//    transpose pass is needed on the way in or out;
//  * the tiles of each phase are spread over one persistent CTA per SM with
//    the LPT greedy ("架构设计" §3.1), cost = k-blocks + epilogue.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <memory>
#include <new>
#include <string>
#include <vector>

#include "../../include/dmuon.h"
#include "host_util.h"
#include "internal.h"

namespace dmuon {

void set_tc_mn_swap(int v);

// Which tensor-core kernel runs the NS phases: 1 = CTA pairs on 256 x 256
// tiles (default), 0 = one CTA per 128 x 256 tile.
static int g_ns_pairs = 1;
// Tile order inside one problem: 1 = longer tile dimension outer, 0 = rows outer.
static int g_tile_order = 1;
// CTA-pair kernel: 1 = symmetric outputs stored as upper blocks only and read
// through transposed loads, 0 = mirrored stores.
static int g_tri = 1;
void set_tc2_variant(int stages, int prefetch);
static int g_tc2_stages_sel = 4, g_tc2_prefetch_sel = 1;
// From the third iteration on (where X is read back in bf16 anyway), fold
// the a*X term of the Combine into the Poly output: B + a I.  1 = on.
static int g_fold_diag = 1;
// CTA-pair kernel: launches whose tiles average fewer 64-deep k-blocks than
// this drain their accumulators with 8 epilogue warps instead of 4.
static int g_epi8_below = 32;
// Momentum overlapped with Newton-Schulz: a large tensor list is cut into
// this many groups with disjoint workspace regions, and group g+1's
// momentum pass (HBM-bound) runs on a side stream while group g's
// Newton-Schulz products (tensor-core-bound) run on the caller's stream.
// 1 = one group, everything on the caller's stream.  A group gets at least
// g_group_min_elems elements (2^30 by default): smaller groups leave their
// launches too few tiles to fill the GPU, which costs more than the hidden
// momentum pass saves (measured: a GPT-2-sized list in 4 groups runs 40 %
// slower, the Llama-3-8B set 1.5 % faster).
static int g_mom_groups = 4;
static int64_t g_group_min_elems = int64_t(1) << 30;
// Slot ranges: 0 = one-group step, 1.. = overlapped groups, 65.. = host pipeline.
constexpr size_t kSlotOverlap = 1, kSlotHost = 65;

// ------------------------------------------------------------------ errors
namespace {
thread_local std::string g_last_error;
}

int set_error(int status, const char* msg) {
  g_last_error = msg ? msg : "";
  return status;
}
void clear_error() { g_last_error.clear(); }

static int cuda_fail(cudaError_t e, const char* where) {
  std::string m = std::string(where) + ": " + cudaGetErrorString(e);
  return set_error(DMUON_ERR_CUDA, m.c_str());
}

#define DM_CUDA(call)                                        \
  do {                                                       \
    cudaError_t e_ = (call);                                 \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call);      \
  } while (0)

// ------------------------------------------------------- driver entry point
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

using PointerAttrFn = CUresult (*)(void*, CUpointer_attribute, CUdeviceptr);

static PointerAttrFn get_pointer_attr_fn() {
  static PointerAttrFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuPointerGetAttribute", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PointerAttrFn>(p);
  }
  return fn;
}

// ------------------------------------------------------------- device mem
struct DevBuf {
  void* p = nullptr;
  size_t bytes = 0;
  void release() {
    if (p) cudaFree(p);
    p = nullptr;
    bytes = 0;
  }
};

static int dev_alloc(DevBuf& b, size_t bytes) {
  b.release();
  if (bytes == 0) return DMUON_OK;
  cudaError_t e = cudaMalloc(&b.p, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    b.p = nullptr;
    std::string m = "cudaMalloc(" + std::to_string(bytes) + " bytes) failed: " + cudaGetErrorString(e);
    return set_error(DMUON_ERR_NOMEM, m.c_str());
  }
  b.bytes = bytes;
  return DMUON_OK;
}

template <class T>
static int upload(DevBuf& b, const std::vector<T>& v) {
  int st = dev_alloc(b, std::max<size_t>(v.size() * sizeof(T), 16));
  if (st != DMUON_OK) return st;
  if (!v.empty()) DM_CUDA(cudaMemcpy(b.p, v.data(), v.size() * sizeof(T), cudaMemcpyHostToDevice));
  return DMUON_OK;
}

// Host table uploaded on the caller's stream through a pinned staging copy,
// skipped when the contents did not change since the last upload.
struct StagedTable {
  DevBuf dev;
  void* pinned = nullptr;
  size_t cap = 0;
  cudaEvent_t done = nullptr;
  std::vector<uint8_t> last;
  void release() {
    dev.release();
    if (pinned) cudaFreeHost(pinned);
    pinned = nullptr;
    cap = 0;
    if (done) cudaEventDestroy(done);
    done = nullptr;
    last.clear();
  }
  int put(const void* data, size_t bytes, cudaStream_t st) {
    if (bytes == last.size() && bytes > 0 && memcmp(data, last.data(), bytes) == 0) return DMUON_OK;
    if (bytes > cap) {
      if (done) DM_CUDA(cudaEventSynchronize(done));
      if (pinned) cudaFreeHost(pinned);
      pinned = nullptr;
      cudaError_t e = cudaMallocHost(&pinned, bytes);
      if (e != cudaSuccess) {
        cudaGetLastError();
        pinned = nullptr;
        cap = 0;
        return set_error(DMUON_ERR_NOMEM, "cudaMallocHost for a descriptor table failed");
      }
      cap = bytes;
      int s = dev_alloc(dev, bytes);
      if (s != DMUON_OK) return s;
      last.clear();
    }
    if (!done) DM_CUDA(cudaEventCreateWithFlags(&done, cudaEventDisableTiming));
    DM_CUDA(cudaEventSynchronize(done));  // previous copy out of `pinned` finished
    memcpy(pinned, data, bytes);
    DM_CUDA(cudaMemcpyAsync(dev.p, pinned, bytes, cudaMemcpyHostToDevice, st));
    DM_CUDA(cudaEventRecord(done, st));
    last.assign(static_cast<const uint8_t*>(data), static_cast<const uint8_t*>(data) + bytes);
    return DMUON_OK;
  }
};

// ------------------------------------------------------------------- plan
struct SliceRef {
  int32_t mat;
  int64_t elem_offset;  // offset of the slice inside its tensor
  int32_t cls;
  int32_t z;            // index within the class
};

struct ShapeClass {
  int32_t m, n, count;
  bool tall;            // m > n: Gram is X^T X, last product X B
  bool f32;             // Newton-Schulz in fp32 on CUDA cores (workspace fp32)
  int64_t ld, ldp;      // workspace row pitch (elements) for X and for A/B
  size_t off_x[2], off_a, off_b;  // byte offsets in the workspace
  size_t off_xf, off_af;          // fp32 side copies of X and A (bf16 path only)
  int32_t map_xk[2], map_xmn[2], map_a, map_b, map_a_mn, map_b_mn;
  int32_t map_x_st[2], map_a_st, map_b_st;  // 64 x 32 boxes for TMA stores
};

struct PhaseTiles {
  int32_t n_tiles = 0;
  int32_t n_ctas = 0;
  double mean_kblocks = 0.0;  // mean main-loop length of the tiles (64-deep k-blocks)
  DevBuf tiles, cta_begin;
};

struct MuonPlan {
  std::string key;
  uint64_t ws_epoch = 0;  // workspace allocation the tables point into
  size_t ws_base = 0;     // byte offset of this plan's region in the workspace
  bool fp32 = false;
  std::vector<SliceRef> slices;
  std::vector<ShapeClass> classes;
  std::vector<Chunk> chunks;
  std::vector<int32_t> slice_chunk_begin, slice_chunk_end;
  size_t ws_bytes = 0;
  DevBuf chunks_dev, partials, inv_norm, maps;
  std::vector<Chunk> chunks_f32;  // chunks of the fp32-class slices only
  DevBuf chunks_f32_dev;
  // Problem tables per kind and variant: 0/1 = X in buffer 0/1 (later
  // iterations), 2 = first iteration, 3 = second iteration.  probs: the
  // bf16 classes (tensor cores); probs_f32: the fp32 classes (CUDA cores,
  // variants 0 and 1 only).
  DevBuf probs[3][4], probs_f32[3][2];
  PhaseTiles phase[3];      // one-CTA tensor-core tiles
  PhaseTiles phase2[3];     // CTA-pair tensor-core tiles
  PhaseTiles phase_f32[3];  // fp32 CUDA-core tiles
  void release() {
    chunks_dev.release();
    chunks_f32_dev.release();
    for (auto& k : probs_f32)
      for (auto& p : k) p.release();
    partials.release();
    inv_norm.release();
    maps.release();
    for (auto& k : probs)
      for (auto& p : k) p.release();
    for (auto* ph : {phase, phase2, phase_f32})
      for (int k = 0; k < 3; ++k) {
        ph[k].tiles.release();
        ph[k].cta_begin.release();
        ph[k].n_tiles = ph[k].n_ctas = 0;
      }
    slices.clear();
    classes.clear();
    chunks.clear();
    chunks_f32.clear();
    key.clear();
  }
};

struct AdamPlan {
  std::string key;
  std::vector<Chunk> chunks;
  DevBuf chunks_dev;
  void release() {
    chunks_dev.release();
    chunks.clear();
    key.clear();
  }
};

// One Muon tensor list's cached state: its plan, its per-call pointer table
// and the descriptor bytes that last passed the reachability check.  Slot 0
// serves dmuon_muon_step; the host pipeline gives each of its groups its own
// slot, so consecutive groups never wait on one another's table uploads.
// All slots share the context's workspace (their steps run one after another
// on one stream); a slot whose plan predates the workspace's current
// allocation is rebuilt.
// Copies of one host-buffer step (dmuon_step_host), cached for the
// descriptor arrays they were built from.
struct CopyRun {
  void* dst;
  const void* src;
  size_t bytes;
  uint64_t dst_id, src_id;  // CUDA allocation ids (0 = unknown)
};

struct HostPlan {
  std::vector<uint8_t> key;
  std::vector<std::pair<int, int>> groups;       // [begin, end) of each Muon group
  std::vector<std::vector<CopyRun>> in, out;     // per group
  std::vector<CopyRun> a_in, a_out;              // AdamW tensors
};

struct MuonSlot {
  MuonPlan plan;
  StagedTable table;
  std::vector<uint8_t> checked;
  void release() {
    plan.release();
    table.release();
    checked.clear();
  }
};

// Per-kernel device timing: events recorded around each launch on the
// launching stream, resolved and summed on read.
struct Profiler {
  bool on = false;
  std::vector<cudaEvent_t> pool;
  struct Pending {
    int kind;
    cudaEvent_t a, b;
  };
  std::vector<Pending> pending;
  double ms[DMUON_KERNEL_KINDS] = {};
  int64_t count[DMUON_KERNEL_KINDS] = {};
  cudaEvent_t get() {
    if (!pool.empty()) {
      cudaEvent_t e = pool.back();
      pool.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    return e;
  }
  void release() {
    for (auto& p : pending) {
      cudaEventDestroy(p.a);
      cudaEventDestroy(p.b);
    }
    pending.clear();
    for (auto e : pool) cudaEventDestroy(e);
    pool.clear();
  }
};

}  // namespace dmuon

struct dmuon_context {
  int device = 0;
  bool dev_ready = false;
  int num_sms = 0;
  int64_t launches = 0;
  dmuon::DevBuf err;
  dmuon::DevBuf ws;
  uint64_t ws_epoch = 0;  // bumped whenever ws is reallocated
  std::vector<std::unique_ptr<dmuon::MuonSlot>> slots;
  dmuon::AdamPlan adam;
  dmuon::StagedTable vec_table;
  dmuon::Profiler prof;
  // AdamW descriptor array whose pointers last passed the reachability check.
  std::vector<uint8_t> checked_vecs;
  // Host pipeline: copy streams, events, cached groups and copy lists.
  cudaStream_t h2d = nullptr, d2h = nullptr;
  std::vector<cudaEvent_t> events;
  dmuon::HostPlan host;
  // Overlapped momentum: side stream and its events.
  cudaStream_t side = nullptr;
  std::vector<cudaEvent_t> side_events;
};

namespace dmuon {
namespace {

struct DeviceGuard {
  int prev = -1;
  bool changed = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) {
      if (cudaSetDevice(dev) == cudaSuccess) changed = true;
    }
  }
  ~DeviceGuard() {
    if (changed) cudaSetDevice(prev);
  }
};

bool finite(float x) { return std::isfinite(x); }

int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int ensure_device(dmuon_context* ctx) {
  if (ctx->dev_ready) return DMUON_OK;
  int count = 0;
  cudaError_t e = cudaGetDeviceCount(&count);
  if (e != cudaSuccess || count <= ctx->device) {
    cudaGetLastError();
    return set_error(DMUON_ERR_UNSUPPORTED, "no CUDA device with the context's ordinal");
  }
  cudaDeviceProp prop;
  DM_CUDA(cudaGetDeviceProperties(&prop, ctx->device));
  if (prop.major != 10)
    return set_error(DMUON_ERR_UNSUPPORTED,
                     "device is not of the sm_100 family (this library is built for sm_103a)");
  ctx->num_sms = prop.multiProcessorCount;
  int st = dev_alloc(ctx->err, 16);
  if (st != DMUON_OK) return st;
  DM_CUDA(cudaMemset(ctx->err.p, 0, 16));
  ctx->dev_ready = true;
  return DMUON_OK;
}

// Every pointer a kernel dereferences must be reachable from the context's
// device: its own memory, managed memory, or page-locked host memory mapped
// into the device's address space (on a Grace host the kernels then read and
// write it over NVLink-C2C, with no staging copy).  Pageable host memory and
// another device's memory are refused here, before any launch.
int check_reachable(const dmuon_context* ctx, const void* p, const char* what, int idx) {
  if (!p) return DMUON_OK;
  cudaPointerAttributes at;
  memset(&at, 0, sizeof at);
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    at.type = cudaMemoryTypeUnregistered;
  }
  bool ok = false;
  if (at.type == cudaMemoryTypeDevice) ok = at.device == ctx->device;
  else if (at.type == cudaMemoryTypeManaged) ok = true;
  else if (at.type == cudaMemoryTypeHost) ok = at.devicePointer == p;
  if (ok) return DMUON_OK;
  char buf[200];
  snprintf(buf, sizeof buf,
           "tensor %d: %s pointer is not reachable from device %d (pageable host memory or another "
           "device's memory)", idx, what, ctx->device);
  return set_error(DMUON_ERR_INVALID_ARG, buf);
}

template <class T>
bool same_bytes(const std::vector<uint8_t>& v, const T* a, int n) {
  return v.size() == sizeof(T) * static_cast<size_t>(n) && memcmp(v.data(), a, v.size()) == 0;
}

template <class T>
void keep_bytes(std::vector<uint8_t>& v, const T* a, int n) {
  v.assign(reinterpret_cast<const uint8_t*>(a), reinterpret_cast<const uint8_t*>(a) + sizeof(T) * static_cast<size_t>(n));
}

int check_matrices_reachable(dmuon_context* ctx, std::vector<uint8_t>& checked, const dmuon_matrix* mats,
                             int n) {
  if (same_bytes(checked, mats, n)) return DMUON_OK;
  checked.clear();
  for (int i = 0; i < n; ++i) {
    int st;
    if ((st = check_reachable(ctx, mats[i].master, "master", i)) != DMUON_OK) return st;
    if ((st = check_reachable(ctx, mats[i].momentum, "momentum", i)) != DMUON_OK) return st;
    if ((st = check_reachable(ctx, mats[i].grad, "grad", i)) != DMUON_OK) return st;
    if ((st = check_reachable(ctx, mats[i].param_bf16, "param", i)) != DMUON_OK) return st;
  }
  keep_bytes(checked, mats, n);
  return DMUON_OK;
}

int check_vectors_reachable(dmuon_context* ctx, const dmuon_vector* ts, int n) {
  if (same_bytes(ctx->checked_vecs, ts, n)) return DMUON_OK;
  ctx->checked_vecs.clear();
  for (int i = 0; i < n; ++i) {
    if (ts[i].numel == 0) continue;
    int st;
    if ((st = check_reachable(ctx, ts[i].master, "master", i)) != DMUON_OK) return st;
    if ((st = check_reachable(ctx, ts[i].exp_avg, "exp_avg", i)) != DMUON_OK) return st;
    if ((st = check_reachable(ctx, ts[i].exp_avg_sq, "exp_avg_sq", i)) != DMUON_OK) return st;
    if ((st = check_reachable(ctx, ts[i].grad, "grad", i)) != DMUON_OK) return st;
    if ((st = check_reachable(ctx, ts[i].param_bf16, "param", i)) != DMUON_OK) return st;
  }
  keep_bytes(ctx->checked_vecs, ts, n);
  return DMUON_OK;
}

int validate_matrix(const dmuon_matrix& M, int idx) {
  char buf[160];
  if (M.rank < 2) {
    snprintf(buf, sizeof buf, "tensor %d has rank %d; Muon needs rank >= 2 (route it to AdamW)", idx, M.rank);
    return set_error(DMUON_ERR_RANK_LT2, buf);
  }
  if (M.rank > 4) {
    snprintf(buf, sizeof buf, "tensor %d has rank %d > 4", idx, M.rank);
    return set_error(DMUON_ERR_SHAPE, buf);
  }
  int64_t numel = 1;
  for (int d = 0; d < M.rank; ++d) {
    if (M.shape[d] < 1 || M.shape[d] > (int64_t(1) << 31)) {
      snprintf(buf, sizeof buf, "tensor %d: dimension %d is %lld", idx, d, (long long)M.shape[d]);
      return set_error(DMUON_ERR_SHAPE, buf);
    }
    numel *= M.shape[d];
    if (numel > (int64_t(1) << 40)) {
      snprintf(buf, sizeof buf, "tensor %d: more than 2^40 elements", idx);
      return set_error(DMUON_ERR_SHAPE, buf);
    }
  }
  const int64_t m = M.shape[M.rank - 2], n = M.shape[M.rank - 1];
  if (m * n >= (int64_t(1) << 31) || m > 65535 * kTcBM || n > 65535 * kTcBM) {
    snprintf(buf, sizeof buf, "tensor %d: a %lld x %lld slice is too large", idx, (long long)m, (long long)n);
    return set_error(DMUON_ERR_SHAPE, buf);
  }
  if (!M.master || !M.momentum || !M.grad) {
    snprintf(buf, sizeof buf, "tensor %d: null master, momentum or grad pointer", idx);
    return set_error(DMUON_ERR_INVALID_ARG, buf);
  }
  if (M.grad_dtype != DMUON_DTYPE_F32 && M.grad_dtype != DMUON_DTYPE_BF16) {
    snprintf(buf, sizeof buf, "tensor %d: grad dtype %d", idx, M.grad_dtype);
    return set_error(DMUON_ERR_DTYPE, buf);
  }
  return DMUON_OK;
}

std::string plan_key(const dmuon_matrix* mats, int n, bool fp32) {
  std::string k = fp32 ? "f32|" : "bf16|";
  k += "o" + std::to_string(g_tile_order) + "|";
  for (int i = 0; i < n; ++i) {
    k += std::to_string(mats[i].rank);
    for (int d = 0; d < mats[i].rank; ++d) k += ":" + std::to_string(mats[i].shape[d]);
    k += ";";
  }
  return k;
}

int make_map(EncodeTiledFn enc, CUtensorMap* out, void* base, int64_t inner, int64_t rows,
             int64_t count, int64_t ld, uint32_t box_inner, uint32_t box_rows) {
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)count};
  cuuint64_t strides[2] = {(cuuint64_t)(ld * 2), (cuuint64_t)(rows * ld * 2)};
  cuuint32_t box[3] = {box_inner, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[200];
    snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled failed (%d) for a %lld x %lld x %lld map", (int)r,
             (long long)inner, (long long)rows, (long long)count);
    return set_error(DMUON_ERR_CUDA, buf);
  }
  return DMUON_OK;
}

// Build the tile list of one phase and balance it over persistent CTAs.
// Tile geometry: 0 = fp32 CUDA-core tiles, 1 = one-CTA tcgen05 tiles,
// 2 = CTA-pair tcgen05 tiles.  `slots` = persistent CTAs (or CTA pairs).
int build_phase_tiles(const std::vector<NsProblem>& probs, int geometry, int slots, PhaseTiles& out) {
  const bool fp32 = geometry == 0;
  const int bm = geometry == 0 ? kSimtBM : geometry == 1 ? kTcBM : kTc2Tile;
  const int bn = geometry == 0 ? kSimtBN : geometry == 1 ? kTcBN : kTc2Tile;
  std::vector<uint2> tiles;
  std::vector<int64_t> cost;
  for (size_t p = 0; p < probs.size(); ++p) {
    const NsProblem& P = probs[p];
    const int tm = (P.M + bm - 1) / bm, tn = (P.N + bn - 1) / bn;
    const int64_t c = (P.K + kTcBK - 1) / kTcBK + 2;
    // Tiles of equal cost run in list order, so consecutive tiles run at the
    // same time: walk the longer tile dimension in the outer loop, so a wave
    // shares few panels of the larger operand (which then stay in L2).
    const bool n_outer = g_tile_order && tn > tm;
    for (int a = 0; a < (n_outer ? tn : tm); ++a)
      for (int b = 0; b < (n_outer ? tm : tn); ++b) {
        const int i = n_outer ? b : a, j = n_outer ? a : b;
        if (P.sym && (i * bm) / bn > j) continue;  // below the diagonal: mirrored
        tiles.push_back(make_uint2(static_cast<uint32_t>(p), (static_cast<uint32_t>(i) << 16) | static_cast<uint32_t>(j)));
        cost.push_back(c);
      }
  }
  out.n_tiles = static_cast<int32_t>(tiles.size());
  double kb = 0.0;
  for (int64_t c : cost) kb += static_cast<double>(c - 2);
  out.mean_kblocks = tiles.empty() ? 0.0 : kb / static_cast<double>(tiles.size());
  if (fp32) {
    out.n_ctas = out.n_tiles;
    int st = upload(out.tiles, tiles);
    if (st != DMUON_OK) return st;
    return upload(out.cta_begin, std::vector<int32_t>{0, out.n_tiles});
  }
  const int R = std::max(1, std::min(slots, out.n_tiles));
  std::vector<int32_t> slot(tiles.size());
  std::vector<int32_t> order;
  int st = lpt_assign_impl(cost.data(), out.n_tiles, R, slot.data(), nullptr, &order);
  if (st != DMUON_OK) return st;
  std::vector<int32_t> counts(static_cast<size_t>(R) + 1, 0);
  for (int32_t t = 0; t < out.n_tiles; ++t) counts[static_cast<size_t>(slot[t]) + 1]++;
  for (int r = 0; r < R; ++r) counts[r + 1] += counts[r];
  std::vector<int32_t> fill(counts.begin(), counts.end() - 1);
  std::vector<uint2> ordered(tiles.size());
  for (int32_t t : order) ordered[static_cast<size_t>(fill[slot[t]]++)] = tiles[static_cast<size_t>(t)];
  out.n_ctas = R;
  st = upload(out.tiles, ordered);
  if (st != DMUON_OK) return st;
  return upload(out.cta_begin, counts);
}

// Slices, shape classes and the workspace layout of a plan, its regions
// starting `ws_base` bytes into the workspace (no device work).
int layout_plan(MuonPlan& P, const dmuon_matrix* mats, int n, bool fp32, size_t ws_base) {
  P.release();
  P.fp32 = fp32;
  P.ws_base = ws_base;

  // Slices and shape classes.
  for (int i = 0; i < n; ++i) {
    const dmuon_matrix& M = mats[i];
    const int32_t m = static_cast<int32_t>(M.shape[M.rank - 2]);
    const int32_t nn = static_cast<int32_t>(M.shape[M.rank - 1]);
    int64_t lead = 1;
    for (int d = 0; d < M.rank - 2; ++d) lead *= M.shape[d];
    int cls = -1;
    for (size_t c = 0; c < P.classes.size(); ++c)
      if (P.classes[c].m == m && P.classes[c].n == nn) cls = static_cast<int>(c);
    if (cls < 0) {
      ShapeClass C{};
      C.m = m;
      C.n = nn;
      C.count = 0;
      C.tall = m > nn;
      C.f32 = fp32 || std::min(m, nn) < kFp32BelowP;
      P.classes.push_back(C);
      cls = static_cast<int>(P.classes.size()) - 1;
    }
    for (int64_t s = 0; s < lead; ++s) {
      SliceRef r;
      r.mat = i;
      r.elem_offset = s * static_cast<int64_t>(m) * nn;
      r.cls = cls;
      r.z = P.classes[static_cast<size_t>(cls)].count++;
      P.slices.push_back(r);
    }
  }
  if (P.slices.size() > (size_t(1) << 30)) return set_error(DMUON_ERR_SHAPE, "too many slices");

  // Workspace layout: per class X0, X1 [count, m, ld] and A, B [count, p, ldp].
  size_t off = ws_base;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += (bytes + 1023) & ~size_t(1023);
    return o;
  };
  for (auto& C : P.classes) {
    const int64_t p = std::min(C.m, C.n);
    const int64_t es = C.f32 ? 4 : 2;
    C.ld = round_up(C.n, 8);
    C.ldp = round_up(p, 8);
    for (int t = 0; t < 2; ++t) C.off_x[t] = take(static_cast<size_t>(C.count) * C.m * C.ld * es);
    C.off_a = take(static_cast<size_t>(C.count) * p * C.ldp * es);
    C.off_b = take(static_cast<size_t>(C.count) * p * C.ldp * es);
    C.off_xf = C.f32 ? 0 : take(static_cast<size_t>(C.count) * C.m * C.ld * 4);
    C.off_af = C.f32 ? 0 : take(static_cast<size_t>(C.count) * p * C.ldp * 4);
  }
  P.ws_bytes = std::max<size_t>(off - ws_base, 1024);
  return DMUON_OK;
}

// Workspace bytes a plan for this tensor list needs.
size_t plan_ws_bytes(const dmuon_matrix* mats, int n, bool fp32) {
  MuonPlan tmp;
  if (layout_plan(tmp, mats, n, fp32, 0) != DMUON_OK) return 0;
  return tmp.ws_bytes;
}

// Grow the workspace to at least `bytes` (every plan built before then
// points into the old allocation and is rebuilt on its next use).
int ensure_workspace(dmuon_context* ctx, size_t bytes) {
  if (ctx->ws.bytes >= bytes) return DMUON_OK;
  ctx->ws.release();
  ctx->ws_epoch++;
  return dev_alloc(ctx->ws, bytes);
}

int build_muon_plan(dmuon_context* ctx, MuonPlan& P, const dmuon_matrix* mats, int n, bool fp32,
                    const std::string& key, size_t ws_base) {
  int st = layout_plan(P, mats, n, fp32, ws_base);
  if (st != DMUON_OK) return st;
  st = ensure_workspace(ctx, P.ws_base + P.ws_bytes);
  if (st != DMUON_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(ctx->ws.p);

  // Chunk table of the streaming passes.
  P.slice_chunk_begin.resize(P.slices.size());
  P.slice_chunk_end.resize(P.slices.size());
  for (size_t s = 0; s < P.slices.size(); ++s) {
    const ShapeClass& C = P.classes[static_cast<size_t>(P.slices[s].cls)];
    const int64_t numel = static_cast<int64_t>(C.m) * C.n;
    P.slice_chunk_begin[s] = static_cast<int32_t>(P.chunks.size());
    for (int64_t st = 0; st < numel; st += kChunkElems) {
      Chunk ch;
      ch.slice = static_cast<int32_t>(s);
      ch.start = st;
      ch.count = static_cast<int32_t>(std::min<int64_t>(kChunkElems, numel - st));
      P.chunks.push_back(ch);
      if (C.f32) P.chunks_f32.push_back(ch);
    }
    P.slice_chunk_end[s] = static_cast<int32_t>(P.chunks.size());
  }
  if (P.chunks.size() > size_t(INT32_MAX)) return set_error(DMUON_ERR_SHAPE, "too many chunks");
  st = upload(P.chunks_dev, P.chunks);
  if (st != DMUON_OK) return st;
  if (!P.chunks_f32.empty()) {
    st = upload(P.chunks_f32_dev, P.chunks_f32);
    if (st != DMUON_OK) return st;
  }
  st = dev_alloc(P.partials, std::max<size_t>(P.chunks.size(), 1) * sizeof(float));
  if (st != DMUON_OK) return st;
  st = dev_alloc(P.inv_norm, std::max<size_t>(P.slices.size(), 1) * sizeof(float));
  if (st != DMUON_OK) return st;

  // Tensor maps (tcgen05 path): per class X0/X1 K-major and MN-major, A, B.
  std::vector<CUtensorMap> maps;
  bool any_bf16 = false;
  for (const auto& C : P.classes) any_bf16 = any_bf16 || !C.f32;
  if (any_bf16) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return set_error(DMUON_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    for (auto& C : P.classes) {
      if (C.f32) continue;
      const int64_t p = std::min(C.m, C.n);
      for (int t = 0; t < 2; ++t) {
        CUtensorMap mk, mm;
        st = make_map(enc, &mk, ws + C.off_x[t], C.n, C.m, C.count, C.ld, 64, 128);
        if (st != DMUON_OK) return st;
        st = make_map(enc, &mm, ws + C.off_x[t], C.n, C.m, C.count, C.ld, 64, 64);
        if (st != DMUON_OK) return st;
        C.map_xk[t] = static_cast<int32_t>(maps.size());
        maps.push_back(mk);
        C.map_xmn[t] = static_cast<int32_t>(maps.size());
        maps.push_back(mm);
      }
      CUtensorMap ma, mb;
      st = make_map(enc, &ma, ws + C.off_a, p, p, C.count, C.ldp, 64, 128);
      if (st != DMUON_OK) return st;
      st = make_map(enc, &mb, ws + C.off_b, p, p, C.count, C.ldp, 64, 128);
      if (st != DMUON_OK) return st;
      C.map_a = static_cast<int32_t>(maps.size());
      maps.push_back(ma);
      C.map_b = static_cast<int32_t>(maps.size());
      maps.push_back(mb);
      // M/N-contiguous views of A and B (64 x 64 boxes): the transposed reads
      // of the CTA-pair kernel's upper-block-only symmetric operands.
      CUtensorMap mat, mbt;
      st = make_map(enc, &mat, ws + C.off_a, p, p, C.count, C.ldp, 64, 64);
      if (st != DMUON_OK) return st;
      st = make_map(enc, &mbt, ws + C.off_b, p, p, C.count, C.ldp, 64, 64);
      if (st != DMUON_OK) return st;
      C.map_a_mn = static_cast<int32_t>(maps.size());
      maps.push_back(mat);
      C.map_b_mn = static_cast<int32_t>(maps.size());
      maps.push_back(mbt);
      // 64 x 32 store boxes: one epilogue warp's 32 rows x 64 columns.
      CUtensorMap st_map;
      for (int t = 0; t < 2; ++t) {
        st = make_map(enc, &st_map, ws + C.off_x[t], C.n, C.m, C.count, C.ld, 64, 32);
        if (st != DMUON_OK) return st;
        C.map_x_st[t] = static_cast<int32_t>(maps.size());
        maps.push_back(st_map);
      }
      st = make_map(enc, &st_map, ws + C.off_a, p, p, C.count, C.ldp, 64, 32);
      if (st != DMUON_OK) return st;
      C.map_a_st = static_cast<int32_t>(maps.size());
      maps.push_back(st_map);
      st = make_map(enc, &st_map, ws + C.off_b, p, p, C.count, C.ldp, 64, 32);
      if (st != DMUON_OK) return st;
      C.map_b_st = static_cast<int32_t>(maps.size());
      maps.push_back(st_map);
    }
    st = upload(P.maps, maps);
    if (st != DMUON_OK) return st;
  }

  // Problems of the three phases.  bf16 classes, variant 0/1: X in buffer
  // 0/1, everything bf16.  Variant 2 (first iteration, X in buffer 0) and 3
  // (second iteration, X in buffer 1) add the fp32 side copies: the first
  // Gram also writes A in fp32, the first Poly reads that fp32 A, the first
  // Combine reads the fp32 X0 and writes X1 in fp32 over it (each element is
  // read before it is written, by the same thread), and the second Combine
  // reads that fp32 X1.  fp32 classes (all of them in validation mode) go to
  // separate lists with variants 0/1 only.
  std::vector<NsProblem> var[3][4], var_f32[3][2];
  for (size_t s_i = 0; s_i < P.slices.size(); ++s_i) {
    const SliceRef& R = P.slices[s_i];
    const ShapeClass& C = P.classes[static_cast<size_t>(R.cls)];
    const int64_t es = C.f32 ? 4 : 2;
    const int32_t p = std::min(C.m, C.n), q = std::max(C.m, C.n);
    const size_t xoff = static_cast<size_t>(R.z) * C.m * C.ld;
    const size_t poff = static_cast<size_t>(R.z) * p * C.ldp;
    uint8_t* A = ws + C.off_a + poff * es;
    uint8_t* B = ws + C.off_b + poff * es;
    float* Xf = C.f32 ? nullptr : reinterpret_cast<float*>(ws + C.off_xf) + xoff;
    float* Af = C.f32 ? nullptr : reinterpret_cast<float*>(ws + C.off_af) + poff;
    for (int par = 0; par < 2; ++par) {
      uint8_t* X = ws + C.off_x[par] + xoff * es;
      uint8_t* Xn = ws + C.off_x[par ^ 1] + xoff * es;
      NsProblem g{}, y{}, c{};
      g.slice = y.slice = c.slice = static_cast<int32_t>(s_i);
      g.z = y.z = c.z = R.z;
      // Gram: p x p, K = q.
      g.M = g.N = p;
      g.K = q;
      g.a = g.b = X;
      g.out = A;
      g.ld_out = C.ldp;
      g.map_out = C.map_a_st;
      if (!C.tall) {  // A = X X^T: A_op(i,k) = X[i,k], B_op(k,j) = X[j,k]
        g.a_si = C.ld; g.a_sk = 1; g.b_sk = 1; g.b_sj = C.ld;
        g.map_a = g.map_b = C.map_xk[par];
        g.majors = 0;
      } else {        // A = X^T X: A_op(i,k) = X[k,i], B_op(k,j) = X[k,j]
        g.a_si = 1; g.a_sk = C.ld; g.b_sk = C.ld; g.b_sj = 1;
        g.map_a = g.map_b = C.map_xmn[par];
        g.majors = 3;
      }
      // Poly: B = b A + c A A, A symmetric so B_op(k,j) = A[k,j] = A[j,k].
      y.M = y.N = y.K = p;
      y.a = y.b = A;
      y.a_si = C.ldp; y.a_sk = 1; y.b_sk = C.ldp; y.b_sj = 1;
      y.map_a = y.map_b = C.map_a;
      y.majors = 0;
      y.tri = 3;
      y.map_a_t = y.map_b_t = C.map_a_mn;
      y.out = B;
      y.ld_out = C.ldp;
      y.map_out = C.map_b_st;
      y.aux = A;
      y.ld_aux = C.ldp;
      g.sym = y.sym = C.f32 ? 0 : 1;
      // Combine: X' = a X + B X (wide) or a X + X B (tall).
      c.out = Xn;
      c.ld_out = C.ld;
      c.map_out = C.map_x_st[par ^ 1];
      c.aux = X;
      c.ld_aux = C.ld;
      if (!C.tall) {  // M = p, N = q, K = p: A_op = B, B_op(k,j) = X[k,j]
        c.M = p; c.N = q; c.K = p;
        c.a = B; c.a_si = C.ldp; c.a_sk = 1;
        c.b = X; c.b_sk = C.ld; c.b_sj = 1;
        c.map_a = C.map_b;
        c.map_b = C.map_xmn[par];
        c.majors = 2;
        c.tri = 1;
        c.map_a_t = C.map_b_mn;
      } else {        // M = q, N = p, K = p: A_op = X, B_op(k,j) = B[k,j] = B[j,k]
        c.M = q; c.N = p; c.K = p;
        c.a = X; c.a_si = C.ld; c.a_sk = 1;
        c.b = B; c.b_sk = C.ldp; c.b_sj = 1;
        c.map_a = C.map_xk[par];
        c.map_b = C.map_b;
        c.majors = 0;
        c.tri = 2;
        c.map_b_t = C.map_b_mn;
      }
      if (C.f32) {
        var_f32[kGram][par].push_back(g);
        var_f32[kPoly][par].push_back(y);
        var_f32[kCombine][par].push_back(c);
        continue;
      }
      var[kGram][par].push_back(g);
      var[kPoly][par].push_back(y);
      var[kCombine][par].push_back(c);
      if (par == 0) {
        g.out2 = Af;
        g.ld_out2 = C.ldp;
        y.aux = Af;
        c.aux = Xf;
        c.out2 = Xf;
        c.ld_out2 = C.ld;
      }
      if (par == 1) c.aux = Xf;
      var[kGram][2 + par].push_back(g);
      var[kPoly][2 + par].push_back(y);
      var[kCombine][2 + par].push_back(c);
    }
  }
  for (int kind = 0; kind < 3; ++kind) {
    for (int v = 0; v < 4; ++v) {
      st = upload(P.probs[kind][v], var[kind][v]);
      if (st != DMUON_OK) return st;
    }
    for (int v = 0; v < 2; ++v) {
      st = upload(P.probs_f32[kind][v], var_f32[kind][v]);
      if (st != DMUON_OK) return st;
    }
  }
  for (int kind = 0; kind < 3; ++kind) {
    if (!var_f32[kind][0].empty()) {
      st = build_phase_tiles(var_f32[kind][0], 0, ctx->num_sms, P.phase_f32[kind]);
      if (st != DMUON_OK) return st;
    }
    if (!var[kind][0].empty()) {
      st = build_phase_tiles(var[kind][0], 1, ctx->num_sms, P.phase[kind]);
      if (st != DMUON_OK) return st;
      const int pairs = std::max(1, std::min(ctx->num_sms / 2, ns_tc2_max_pairs()));
      st = build_phase_tiles(var[kind][0], 2, pairs, P.phase2[kind]);
      if (st != DMUON_OK) return st;
    }
  }
  P.key = key;
  P.ws_epoch = ctx->ws_epoch;
  return DMUON_OK;
}

// Run one launch, counting it and (when profiling) bracketing it with events.
template <class F>
int timed_launch(dmuon_context* ctx, int kind, cudaStream_t s, F&& launch) {
  Profiler& P = ctx->prof;
  cudaEvent_t a = nullptr, b = nullptr;
  if (P.on) {
    a = P.get();
    b = P.get();
    if (a) cudaEventRecord(a, s);
  }
  cudaError_t e = launch();
  if (e != cudaSuccess) {
    if (a) P.pool.push_back(a);
    if (b) P.pool.push_back(b);
    return cuda_fail(e, "kernel launch");
  }
  ctx->launches++;
  if (P.on && a && b) {
    cudaEventRecord(b, s);
    P.pending.push_back({kind, a, b});
  }
  return DMUON_OK;
}

// Argument checks of a Muon step (host only, before any CUDA call).
int validate_muon_call(const dmuon_matrix* mats, int32_t n, float lr, float momentum, float wd,
                       int32_t ns_steps, float a, float b, float c, uint32_t flags) {
  if (n < 0 || (n > 0 && !mats)) return set_error(DMUON_ERR_INVALID_ARG, "muon_step: bad tensor list");
  if (!finite(lr) || !finite(momentum) || !finite(wd) || !finite(a) || !finite(b) || !finite(c))
    return set_error(DMUON_ERR_INVALID_ARG, "muon_step: non-finite hyper-parameter");
  if (ns_steps < 0 || ns_steps > 100) return set_error(DMUON_ERR_INVALID_ARG, "muon_step: ns_steps outside [0, 100]");
  if (flags & ~uint32_t(DMUON_FLAG_NESTEROV | DMUON_FLAG_FP32_NS))
    return set_error(DMUON_ERR_INVALID_ARG, "muon_step: unknown flag bits");
  for (int i = 0; i < n; ++i) {
    int st = validate_matrix(mats[i], i);
    if (st != DMUON_OK) return st;
  }
  return DMUON_OK;
}

// Argument checks of an AdamW step (host only, before any CUDA call).
int validate_adamw_call(const dmuon_vector* ts, int32_t n, float lr, float beta1, float beta2, float eps,
                        float wd, int64_t step) {
  if (n < 0 || (n > 0 && !ts)) return set_error(DMUON_ERR_INVALID_ARG, "adamw_step: bad tensor list");
  if (!finite(lr) || !finite(wd) || !finite(eps) || eps < 0.f || !(beta1 >= 0.f && beta1 < 1.f) ||
      !(beta2 >= 0.f && beta2 < 1.f))
    return set_error(DMUON_ERR_INVALID_ARG, "adamw_step: bad hyper-parameter");
  if (step < 1) return set_error(DMUON_ERR_INVALID_ARG, "adamw_step: step counter must be >= 1");
  for (int i = 0; i < n; ++i) {
    const dmuon_vector& V = ts[i];
    char buf[120];
    if (V.numel < 0 || V.numel > (int64_t(1) << 40)) {
      snprintf(buf, sizeof buf, "adamw tensor %d: numel %lld", i, (long long)V.numel);
      return set_error(DMUON_ERR_SHAPE, buf);
    }
    if (V.numel > 0 && (!V.master || !V.exp_avg || !V.exp_avg_sq || !V.grad)) {
      snprintf(buf, sizeof buf, "adamw tensor %d: null pointer", i);
      return set_error(DMUON_ERR_INVALID_ARG, buf);
    }
    if (V.grad_dtype != DMUON_DTYPE_F32 && V.grad_dtype != DMUON_DTYPE_BF16) {
      snprintf(buf, sizeof buf, "adamw tensor %d: grad dtype %d", i, V.grad_dtype);
      return set_error(DMUON_ERR_DTYPE, buf);
    }
  }
  return DMUON_OK;
}

MuonSlot* get_slot(dmuon_context* ctx, size_t i) {
  while (ctx->slots.size() <= i) {
    MuonSlot* m = new (std::nothrow) MuonSlot();
    if (!m) return nullptr;
    ctx->slots.emplace_back(m);
  }
  return ctx->slots[i].get();
}

// The slot's plan for this tensor list, rebuilt when the shapes or its
// workspace region changed or the workspace was reallocated since.
int prepare_slot(dmuon_context* ctx, MuonSlot& S, const dmuon_matrix* mats, int n, bool fp32,
                 size_t ws_base = 0) {
  const std::string key = plan_key(mats, n, fp32);
  if (key == S.plan.key && S.plan.ws_epoch == ctx->ws_epoch && S.plan.ws_base == ws_base) return DMUON_OK;
  int st = build_muon_plan(ctx, S.plan, mats, n, fp32, key, ws_base);
  if (st != DMUON_OK) S.plan.release();
  return st;
}

// Stage 1 of a Muon step on a prepared slot: the per-call pointer table,
// uploaded on stream s.
int muon_stage_table(dmuon_context* ctx, MuonSlot& S, const dmuon_matrix* mats, int n, int32_t ns_steps,
                     cudaStream_t s) {
  int st = check_matrices_reachable(ctx, S.checked, mats, n);
  if (st != DMUON_OK) return st;
  MuonPlan& P = S.plan;
  uint8_t* ws = static_cast<uint8_t*>(ctx->ws.p);

  // Per-call pointer table.
  std::vector<SliceDesc> table(P.slices.size());
  for (size_t i = 0; i < P.slices.size(); ++i) {
    const SliceRef& R = P.slices[i];
    const ShapeClass& C = P.classes[static_cast<size_t>(R.cls)];
    const dmuon_matrix& M = mats[R.mat];
    SliceDesc& D = table[i];
    memset(&D, 0, sizeof D);
    D.master = M.master + R.elem_offset;
    D.momentum = M.momentum + R.elem_offset;
    D.grad_bf16 = M.grad_dtype == DMUON_DTYPE_BF16;
    D.grad = static_cast<const uint8_t*>(M.grad) + R.elem_offset * (D.grad_bf16 ? 2 : 4);
    D.param = M.param_bf16 ? M.param_bf16 + R.elem_offset : nullptr;
    const size_t xoff = static_cast<size_t>(R.z) * C.m * C.ld * (C.f32 ? 4 : 2);
    D.x0 = ws + C.off_x[0] + xoff;
    D.x0f = C.f32 ? nullptr : reinterpret_cast<float*>(ws + C.off_xf) + static_cast<size_t>(R.z) * C.m * C.ld;
    D.x_f32 = C.f32 ? 1 : 0;
    D.xk = ws + C.off_x[ns_steps & 1] + xoff;
    D.ld = C.ld;
    D.m = C.m;
    D.n = C.n;
    D.vec_ok = (C.n % 8 == 0) && aligned16(D.master) && aligned16(D.momentum) &&
               aligned16(D.grad) && (!D.param || aligned16(D.param));
    D.shape_scale = static_cast<float>(std::sqrt(std::max(1.0, double(C.m) / double(C.n))));
    D.chunk_begin = P.slice_chunk_begin[i];
    D.chunk_end = P.slice_chunk_end[i];
  }
  return S.table.put(table.data(), table.size() * sizeof(SliceDesc), s);
}

// Stage 2: momentum pass and per-slice norms (needs stage 1 on s).
int muon_launch_front(dmuon_context* ctx, MuonSlot& S, float momentum, uint32_t flags, cudaStream_t s) {
  MuonPlan& P = S.plan;
  const SliceDesc* d_slices = static_cast<const SliceDesc*>(S.table.dev.p);
  const Chunk* d_chunks = static_cast<const Chunk*>(P.chunks_dev.p);
  float* partials = static_cast<float*>(P.partials.p);
  float* inv_norm = static_cast<float*>(P.inv_norm.p);
  const int n_chunks = static_cast<int>(P.chunks.size());
  const int nesterov = (flags & DMUON_FLAG_NESTEROV) ? 1 : 0;
  int st = timed_launch(ctx, DMUON_KERNEL_MOMENTUM, s, [&] {
    return launch_momentum(d_slices, d_chunks, n_chunks, momentum, nesterov, 0, partials, s);
  });
  if (st != DMUON_OK) return st;
  return timed_launch(ctx, DMUON_KERNEL_NORM, s, [&] {
    return launch_norm(d_slices, static_cast<int>(P.slices.size()), partials, inv_norm, s);
  });
}

// Stage 3: the Newton-Schulz launches and the update (needs stage 2's
// results, ordered before s).
int muon_launch_ns(dmuon_context* ctx, MuonSlot& S, float lr, float wd, int32_t ns_steps, float a, float b,
                   float c, cudaStream_t s) {
  MuonPlan& P = S.plan;
  const SliceDesc* d_slices = static_cast<const SliceDesc*>(S.table.dev.p);
  const Chunk* d_chunks = static_cast<const Chunk*>(P.chunks_dev.p);
  float* inv_norm = static_cast<float*>(P.inv_norm.p);
  const int n_chunks = static_cast<int>(P.chunks.size());
  int st = DMUON_OK;
  for (int it = 0; it < ns_steps; ++it) {
    const int variant = it < 2 ? 2 + it : (it & 1);
    for (int kind = kGram; kind <= kCombine; ++kind) {
      NsLaunch L{};
      L.maps = static_cast<const CUtensorMap*>(P.maps.p);
      L.gscale = (it == 0 && kind != kPoly) ? inv_norm : nullptr;
      L.gpow = (kind == kGram) ? 2 : 1;
      L.kind = kind;
      L.a = a;
      L.b = b;
      L.c = c;
      L.err = static_cast<int*>(ctx->err.p);
      // Tensor-core launch over the bf16 classes.
      if (P.phase[kind].n_tiles > 0) {
        NsLaunch T = L;
        T.probs = static_cast<const NsProblem*>(P.probs[kind][variant].p);
        T.aux_f32 = ((it == 0 && kind != kGram) || (it == 1 && kind == kCombine)) ? 1 : 0;
        if (g_fold_diag && it >= 2) {
          // X' = a X + B X = (a I + B) X: the Poly adds a on B's diagonal and
          // the Combine reads no aux.
          if (kind == kPoly) T.diag = a;
          if (kind == kCombine) T.a = 0.f;
        }
        if (kind == kCombine && it == ns_steps - 1) {
          // The last Combine applies the update itself (no X store, no update pass).
          T.fuse_update = 1;
          T.slices = d_slices;
          T.lr = lr;
          T.wd = wd;
        }
        const bool pairs = g_ns_pairs != 0;
        T.tri = (pairs && g_tri) ? 1 : 0;
        const PhaseTiles& PT = pairs ? P.phase2[kind] : P.phase[kind];
        T.epi8 = (!T.fuse_update && PT.mean_kblocks < static_cast<double>(g_epi8_below)) ? 1 : 0;
        T.tiles = static_cast<const uint2*>(PT.tiles.p);
        T.cta_begin = static_cast<const int32_t*>(PT.cta_begin.p);
        st = timed_launch(ctx, DMUON_KERNEL_NS_GRAM + kind, s, [&] {
          return pairs ? launch_ns_tc2(T, PT.n_ctas, s) : launch_ns_tc(T, PT.n_ctas, s);
        });
        if (st != DMUON_OK) return st;
      }
      // CUDA-core launch over the fp32 classes.
      const PhaseTiles& PF = P.phase_f32[kind];
      if (PF.n_tiles > 0) {
        NsLaunch F = L;
        F.probs = static_cast<const NsProblem*>(P.probs_f32[kind][it & 1].p);
        F.tiles = static_cast<const uint2*>(PF.tiles.p);
        F.cta_begin = static_cast<const int32_t*>(PF.cta_begin.p);
        st = timed_launch(ctx, DMUON_KERNEL_NS_GRAM + kind, s, [&] { return launch_ns_simt(F, PF.n_tiles, s); });
        if (st != DMUON_OK) return st;
      }
    }
  }
  // The bf16 classes' update is fused into their last Combine; the update
  // pass covers the fp32 classes (every slice when there are no iterations).
  const bool all = ns_steps == 0;
  const int n_upd = all ? n_chunks : static_cast<int>(P.chunks_f32.size());
  if (n_upd == 0) return DMUON_OK;
  const Chunk* d_upd = all ? d_chunks : static_cast<const Chunk*>(P.chunks_f32_dev.p);
  return timed_launch(ctx, DMUON_KERNEL_UPDATE, s, [&] {
    return launch_update(d_slices, d_upd, n_upd, lr, wd, 0, all ? inv_norm : nullptr, s);
  });
}

// One Muon step of a validated, non-empty tensor list on the current device,
// every stage on stream s.
int muon_step_impl(dmuon_context* ctx, MuonSlot& S, const dmuon_matrix* mats, int n, float lr,
                   float momentum, float wd, int32_t ns_steps, float a, float b, float c,
                   uint32_t flags, cudaStream_t s) {
  int st = prepare_slot(ctx, S, mats, n, (flags & DMUON_FLAG_FP32_NS) != 0);
  if (st != DMUON_OK) return st;
  st = muon_stage_table(ctx, S, mats, n, ns_steps, s);
  if (st != DMUON_OK) return st;
  st = muon_launch_front(ctx, S, momentum, flags, s);
  if (st != DMUON_OK) return st;
  return muon_launch_ns(ctx, S, lr, wd, ns_steps, a, b, c, s);
}

int64_t matrix_elems(const dmuon_matrix& M) {
  int64_t k = 1;
  for (int d = 0; d < M.rank; ++d) k *= M.shape[d];
  return k;
}

// A Muon step with the momentum of group g+1 overlapping the Newton-Schulz
// launches of group g (groups: consecutive tensors of about equal element
// count, each with its own plan and workspace region).
int muon_step_overlapped(dmuon_context* ctx, const dmuon_matrix* mats, int n, int groups, float lr,
                         float momentum, float wd, int32_t ns_steps, float a, float b, float c,
                         uint32_t flags, cudaStream_t s) {
  const bool fp32 = (flags & DMUON_FLAG_FP32_NS) != 0;
  int64_t total = 0;
  for (int i = 0; i < n; ++i) total += matrix_elems(mats[i]);
  std::vector<std::pair<int, int>> range;
  {
    int start = 0;
    int64_t acc = 0;
    for (int i = 0; i < n; ++i) {
      acc += matrix_elems(mats[i]);
      const int closed = static_cast<int>(range.size());
      if (closed < groups - 1 && i + 1 < n && double(acc) >= double(total) * double(closed + 1) / double(groups)) {
        range.push_back({start, i + 1});
        start = i + 1;
      }
    }
    if (start < n) range.push_back({start, n});
  }
  const int G = static_cast<int>(range.size());
  std::vector<size_t> base(static_cast<size_t>(G));
  size_t off = 0;
  for (int g = 0; g < G; ++g) {
    base[static_cast<size_t>(g)] = off;
    const size_t bytes = plan_ws_bytes(mats + range[static_cast<size_t>(g)].first,
                                       range[static_cast<size_t>(g)].second - range[static_cast<size_t>(g)].first, fp32);
    if (bytes == 0) return set_error(DMUON_ERR_SHAPE, "muon_step: workspace layout failed");
    off += (bytes + 1023) & ~size_t(1023);
  }
  int st = ensure_workspace(ctx, off);
  if (st != DMUON_OK) return st;
  std::vector<MuonSlot*> S(static_cast<size_t>(G));
  for (int g = 0; g < G; ++g) {
    S[static_cast<size_t>(g)] = get_slot(ctx, kSlotOverlap + static_cast<size_t>(g));
    if (!S[static_cast<size_t>(g)]) return set_error(DMUON_ERR_NOMEM, "muon_step: host allocation failed");
    st = prepare_slot(ctx, *S[static_cast<size_t>(g)], mats + range[static_cast<size_t>(g)].first,
                      range[static_cast<size_t>(g)].second - range[static_cast<size_t>(g)].first, fp32,
                      base[static_cast<size_t>(g)]);
    if (st != DMUON_OK) return st;
  }
  if (!ctx->side) DM_CUDA(cudaStreamCreateWithFlags(&ctx->side, cudaStreamNonBlocking));
  while (ctx->side_events.size() < static_cast<size_t>(G) + 2) {
    cudaEvent_t e = nullptr;
    DM_CUDA(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
    ctx->side_events.push_back(e);
  }
  cudaEvent_t fork = ctx->side_events[0], join = ctx->side_events[1];
  DM_CUDA(cudaEventRecord(fork, s));
  DM_CUDA(cudaStreamWaitEvent(ctx->side, fork, 0));
  // Side stream: every group's pointer table, momentum pass and norms.
  for (int g = 0; g < G && st == DMUON_OK; ++g) {
    const int b0 = range[static_cast<size_t>(g)].first, cnt = range[static_cast<size_t>(g)].second - b0;
    st = muon_stage_table(ctx, *S[static_cast<size_t>(g)], mats + b0, cnt, ns_steps, ctx->side);
    if (st == DMUON_OK) st = muon_launch_front(ctx, *S[static_cast<size_t>(g)], momentum, flags, ctx->side);
    if (st == DMUON_OK && cudaEventRecord(ctx->side_events[2 + static_cast<size_t>(g)], ctx->side) != cudaSuccess)
      st = cuda_fail(cudaGetLastError(), "muon_step: event record");
  }
  if (st != DMUON_OK) {
    // Leave `stream` ordered after whatever reached the side stream.
    if (cudaEventRecord(join, ctx->side) == cudaSuccess) cudaStreamWaitEvent(s, join, 0);
    return st;
  }
  // Caller's stream: each group's Newton-Schulz once its momentum is done.
  for (int g = 0; g < G; ++g) {
    DM_CUDA(cudaStreamWaitEvent(s, ctx->side_events[2 + static_cast<size_t>(g)], 0));
    st = muon_launch_ns(ctx, *S[static_cast<size_t>(g)], lr, wd, ns_steps, a, b, c, s);
    if (st != DMUON_OK) return st;
  }
  return DMUON_OK;
}


// One AdamW step of a validated, non-empty tensor list on the current device.
int adamw_step_impl(dmuon_context* ctx, const dmuon_vector* ts, int n, float lr, float beta1, float beta2,
                    float eps, float wd, int64_t step, cudaStream_t s) {
  int st = check_vectors_reachable(ctx, ts, n);
  if (st != DMUON_OK) return st;

  std::string key;
  for (int i = 0; i < n; ++i) key += std::to_string(ts[i].numel) + ";";
  AdamPlan& A = ctx->adam;
  if (key != A.key) {
    A.release();
    for (int i = 0; i < n; ++i)
      for (int64_t e = 0; e < ts[i].numel; e += kChunkElems) {
        Chunk ch;
        ch.slice = i;
        ch.start = e;
        ch.count = static_cast<int32_t>(std::min<int64_t>(kChunkElems, ts[i].numel - e));
        A.chunks.push_back(ch);
      }
    if (A.chunks.size() > size_t(INT32_MAX)) return set_error(DMUON_ERR_SHAPE, "too many chunks");
    st = upload(A.chunks_dev, A.chunks);
    if (st != DMUON_OK) {
      A.release();
      return st;
    }
    A.key = key;
  }
  std::vector<VecDesc> table(static_cast<size_t>(n));
  for (int i = 0; i < n; ++i) {
    VecDesc& D = table[static_cast<size_t>(i)];
    memset(&D, 0, sizeof D);
    D.master = ts[i].master;
    D.exp_avg = ts[i].exp_avg;
    D.exp_avg_sq = ts[i].exp_avg_sq;
    D.grad = ts[i].grad;
    D.param = ts[i].param_bf16;
    D.grad_bf16 = ts[i].grad_dtype == DMUON_DTYPE_BF16;
    D.vec_ok = aligned16(D.master) && aligned16(D.exp_avg) && aligned16(D.exp_avg_sq) &&
               aligned16(D.grad) && (!D.param || aligned16(D.param));
  }
  st = ctx->vec_table.put(table.data(), table.size() * sizeof(VecDesc), s);
  if (st != DMUON_OK) return st;
  const double bc1 = 1.0 - std::pow(double(beta1), double(step));
  const double bc2 = 1.0 - std::pow(double(beta2), double(step));
  return timed_launch(ctx, DMUON_KERNEL_ADAMW, s, [&] {
    return launch_adamw(static_cast<const VecDesc*>(ctx->vec_table.dev.p),
                        static_cast<const Chunk*>(A.chunks_dev.p), static_cast<int>(A.chunks.size()),
                        lr, beta1, beta2, eps, wd, static_cast<float>(bc1),
                        static_cast<float>(std::sqrt(bc2)), s);
  });
}


// ------------------------------------------------------------ host pipeline
// Id of the CUDA allocation holding `p` (0 when the driver does not know it).
uint64_t buffer_id(const void* p) {
  PointerAttrFn fn = get_pointer_attr_fn();
  unsigned long long id = 0;
  if (!fn || !p ||
      fn(&id, CU_POINTER_ATTRIBUTE_BUFFER_ID, static_cast<CUdeviceptr>(reinterpret_cast<uintptr_t>(p))) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Append a copy, merged into the previous one when its source and its
// destination both continue the previous ones inside the same allocations
// (one copy may not span two allocations, however adjacent).
void add_run(std::vector<CopyRun>& runs, void* dst, const void* src, size_t bytes) {
  if (bytes == 0) return;
  const uint64_t did = buffer_id(dst), sid = buffer_id(src);
  if (!runs.empty()) {
    CopyRun& r = runs.back();
    if (static_cast<uint8_t*>(r.dst) + r.bytes == dst && static_cast<const uint8_t*>(r.src) + r.bytes == src &&
        did != 0 && sid != 0 && did == r.dst_id && sid == r.src_id) {
      r.bytes += bytes;
      return;
    }
  }
  runs.push_back({dst, src, bytes, did, sid});
}

int enqueue_runs(const std::vector<CopyRun>& runs, cudaMemcpyKind kind, cudaStream_t st) {
  for (const CopyRun& r : runs) DM_CUDA(cudaMemcpyAsync(r.dst, r.src, r.bytes, kind, st));
  return DMUON_OK;
}

int check_page_locked(const void* p, const char* what, int idx) {
  if (!p) return DMUON_OK;
  cudaPointerAttributes at;
  memset(&at, 0, sizeof at);
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    at.type = cudaMemoryTypeUnregistered;
  }
  if (at.type == cudaMemoryTypeHost) return DMUON_OK;
  char buf[160];
  snprintf(buf, sizeof buf, "tensor %d: %s is not page-locked host memory", idx, what);
  return set_error(DMUON_ERR_INVALID_ARG, buf);
}

int ensure_events(dmuon_context* ctx, size_t count) {
  while (ctx->events.size() < count) {
    cudaEvent_t e = nullptr;
    DM_CUDA(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
    ctx->events.push_back(e);
  }
  return DMUON_OK;
}

int64_t matrix_numel(const dmuon_matrix& M) {
  int64_t k = 1;
  for (int d = 0; d < M.rank; ++d) k *= M.shape[d];
  return k;
}

// Consecutive groups of about equal Newton-Schulz work (element count when
// there are no iterations), every group non-empty.
std::vector<std::pair<int, int>> split_groups(const dmuon_matrix* mats, int n, int groups, int ns_steps) {
  std::vector<double> cost(static_cast<size_t>(n));
  double total = 0.0;
  for (int i = 0; i < n; ++i) {
    const dmuon_matrix& M = mats[i];
    const double m = double(M.shape[M.rank - 2]), q0 = double(M.shape[M.rank - 1]);
    const double p = std::min(m, q0), q = std::max(m, q0);
    const double lead = double(matrix_numel(M)) / (m * q0);
    cost[static_cast<size_t>(i)] = ns_steps > 0 ? lead * (4.0 * p * p * q + 2.0 * p * p * p) : lead * m * q0;
    total += cost[static_cast<size_t>(i)];
  }
  std::vector<std::pair<int, int>> out;
  int start = 0;
  double acc = 0.0;
  for (int i = 0; i < n; ++i) {
    acc += cost[static_cast<size_t>(i)];
    const int closed = static_cast<int>(out.size());
    if (closed < groups - 1 && i + 1 < n && acc >= total * double(closed + 1) / double(groups)) {
      out.push_back({start, i + 1});
      start = i + 1;
    }
  }
  if (start < n) out.push_back({start, n});
  return out;
}

}  // namespace
}  // namespace dmuon

using namespace dmuon;

extern "C" {

const char* dmuon_status_string(int status) {
  switch (status) {
    case DMUON_OK: return "ok";
    case DMUON_ERR_INVALID_ARG: return "invalid argument";
    case DMUON_ERR_RANK_LT2: return "Muon tensor of rank < 2";
    case DMUON_ERR_SHAPE: return "unsupported shape";
    case DMUON_ERR_DTYPE: return "unsupported dtype";
    case DMUON_ERR_CUDA: return "CUDA error";
    case DMUON_ERR_TIMEOUT: return "device-side wait timed out";
    case DMUON_ERR_NOMEM: return "out of memory";
    case DMUON_ERR_UNSUPPORTED: return "unsupported device";
    default: return "unknown status";
  }
}

const char* dmuon_last_error(void) { return g_last_error.c_str(); }

int dmuon_context_create(dmuon_context** out, int32_t device) {
  clear_error();
  if (!out || device < 0) return set_error(DMUON_ERR_INVALID_ARG, "context_create: null out or negative device");
  dmuon_context* c = new (std::nothrow) dmuon_context();
  if (!c) return set_error(DMUON_ERR_NOMEM, "context_create: host allocation failed");
  c->device = device;
  *out = c;
  return DMUON_OK;
}

int dmuon_context_destroy(dmuon_context* ctx) {
  clear_error();
  if (!ctx) return DMUON_OK;
  if (ctx->dev_ready) {
    DeviceGuard g(ctx->device);
    cudaDeviceSynchronize();
    for (auto& sl : ctx->slots) sl->release();
    ctx->slots.clear();
    ctx->adam.release();
    ctx->vec_table.release();
    for (cudaEvent_t e : ctx->events) cudaEventDestroy(e);
    ctx->events.clear();
    for (cudaEvent_t e : ctx->side_events) cudaEventDestroy(e);
    ctx->side_events.clear();
    if (ctx->side) cudaStreamDestroy(ctx->side);
    ctx->side = nullptr;
    if (ctx->h2d) cudaStreamDestroy(ctx->h2d);
    if (ctx->d2h) cudaStreamDestroy(ctx->d2h);
    ctx->h2d = ctx->d2h = nullptr;
    ctx->prof.release();
    ctx->ws.release();
    ctx->err.release();
  }
  delete ctx;
  return DMUON_OK;
}

int64_t dmuon_kernel_launches(const dmuon_context* ctx) { return ctx ? ctx->launches : -1; }

int dmuon_muon_step(dmuon_context* ctx, const dmuon_matrix* mats, int32_t n, float lr,
                    float momentum, float wd, int32_t ns_steps, float a, float b, float c,
                    uint32_t flags, void* stream) {
  clear_error();
  if (!ctx) return set_error(DMUON_ERR_INVALID_ARG, "muon_step: null context");
  int st = validate_muon_call(mats, n, lr, momentum, wd, ns_steps, a, b, c, flags);
  if (st != DMUON_OK || n == 0) return st;
  DeviceGuard guard(ctx->device);
  st = ensure_device(ctx);
  if (st != DMUON_OK) return st;
  int64_t total = 0;
  for (int i = 0; i < n; ++i) total += matrix_elems(mats[i]);
  const int groups = static_cast<int>(std::min<int64_t>({int64_t(g_mom_groups), int64_t(n), total / g_group_min_elems}));
  if (groups > 1)
    return muon_step_overlapped(ctx, mats, n, groups, lr, momentum, wd, ns_steps, a, b, c, flags,
                                static_cast<cudaStream_t>(stream));
  MuonSlot* S = get_slot(ctx, 0);
  if (!S) return set_error(DMUON_ERR_NOMEM, "muon_step: host allocation failed");
  return muon_step_impl(ctx, *S, mats, n, lr, momentum, wd, ns_steps, a, b, c, flags,
                        static_cast<cudaStream_t>(stream));
}

int dmuon_adamw_step(dmuon_context* ctx, const dmuon_vector* ts, int32_t n, float lr, float beta1,
                     float beta2, float eps, float wd, int64_t step, void* stream) {
  clear_error();
  if (!ctx) return set_error(DMUON_ERR_INVALID_ARG, "adamw_step: null context");
  int st = validate_adamw_call(ts, n, lr, beta1, beta2, eps, wd, step);
  if (st != DMUON_OK || n == 0) return st;
  DeviceGuard guard(ctx->device);
  st = ensure_device(ctx);
  if (st != DMUON_OK) return st;
  return adamw_step_impl(ctx, ts, n, lr, beta1, beta2, eps, wd, step, static_cast<cudaStream_t>(stream));
}

int dmuon_step_host(dmuon_context* ctx, const dmuon_matrix* mats, const dmuon_host_io* mat_io, int32_t n_mats,
                    const dmuon_muon_hparams* muon, const dmuon_vector* vecs, const dmuon_host_io* vec_io,
                    int32_t n_vecs, const dmuon_adamw_hparams* adamw, int32_t n_groups, void* stream) {
  clear_error();
  if (!ctx) return set_error(DMUON_ERR_INVALID_ARG, "step_host: null context");
  if (n_mats < 0 || n_vecs < 0 || (n_mats > 0 && (!mats || !mat_io || !muon)) ||
      (n_vecs > 0 && (!vecs || !vec_io || !adamw)))
    return set_error(DMUON_ERR_INVALID_ARG, "step_host: bad tensor list or missing hyper-parameters");
  if (n_groups < 1 || n_groups > 64) return set_error(DMUON_ERR_INVALID_ARG, "step_host: n_groups outside [1, 64]");
  int st;
  if (n_mats > 0) {
    st = validate_muon_call(mats, n_mats, muon->lr, muon->momentum, muon->wd, muon->ns_steps, muon->a, muon->b,
                            muon->c, muon->flags);
    if (st != DMUON_OK) return st;
  }
  if (n_vecs > 0) {
    st = validate_adamw_call(vecs, n_vecs, adamw->lr, adamw->beta1, adamw->beta2, adamw->eps, adamw->wd,
                             adamw->step);
    if (st != DMUON_OK) return st;
  }
  char buf[160];
  for (int i = 0; i < n_mats; ++i) {
    if (!mat_io[i].grad_host || (mat_io[i].param_host && !mats[i].param_bf16)) {
      snprintf(buf, sizeof buf, "step_host: Muon tensor %d: null grad_host, or param_host without param_bf16", i);
      return set_error(DMUON_ERR_INVALID_ARG, buf);
    }
  }
  for (int i = 0; i < n_vecs; ++i) {
    if (vecs[i].numel > 0 && (!vec_io[i].grad_host || (vec_io[i].param_host && !vecs[i].param_bf16))) {
      snprintf(buf, sizeof buf, "step_host: AdamW tensor %d: null grad_host, or param_host without param_bf16", i);
      return set_error(DMUON_ERR_INVALID_ARG, buf);
    }
  }
  if (n_mats == 0 && n_vecs == 0) return DMUON_OK;

  DeviceGuard guard(ctx->device);
  st = ensure_device(ctx);
  if (st != DMUON_OK) return st;
  if (!ctx->h2d) DM_CUDA(cudaStreamCreateWithFlags(&ctx->h2d, cudaStreamNonBlocking));
  if (!ctx->d2h) DM_CUDA(cudaStreamCreateWithFlags(&ctx->d2h, cudaStreamNonBlocking));
  // Groups and copy lists, rebuilt (and the host buffers checked) only when
  // the descriptor arrays change.
  HostPlan& H = ctx->host;
  {
    std::vector<uint8_t> key, part;
    auto append = [&](const std::vector<uint8_t>& b) { key.insert(key.end(), b.begin(), b.end()); };
    keep_bytes(part, mats, n_mats);
    append(part);
    keep_bytes(part, mat_io, n_mats);
    append(part);
    keep_bytes(part, vecs, n_vecs);
    append(part);
    keep_bytes(part, vec_io, n_vecs);
    append(part);
    const int32_t extra[3] = {n_mats, n_groups, n_mats > 0 && muon->ns_steps > 0 ? 1 : 0};
    keep_bytes(part, extra, 3);
    append(part);
    if (key != H.key) {
      H = HostPlan();
      for (int i = 0; i < n_mats; ++i) {
        if ((st = check_page_locked(mat_io[i].grad_host, "grad_host", i)) != DMUON_OK) return st;
        if ((st = check_page_locked(mat_io[i].param_host, "param_host", i)) != DMUON_OK) return st;
      }
      for (int i = 0; i < n_vecs; ++i) {
        if (vecs[i].numel == 0) continue;
        if ((st = check_page_locked(vec_io[i].grad_host, "grad_host", i)) != DMUON_OK) return st;
        if ((st = check_page_locked(vec_io[i].param_host, "param_host", i)) != DMUON_OK) return st;
      }
      H.groups = split_groups(mats, n_mats, n_groups, n_mats > 0 ? muon->ns_steps : 0);
      const size_t G = H.groups.size();
      H.in.resize(G);
      H.out.resize(G);
      auto grad_bytes = [](int64_t numel, int32_t dtype) {
        return static_cast<size_t>(numel) * (dtype == DMUON_DTYPE_BF16 ? 2 : 4);
      };
      for (size_t g = 0; g < G; ++g)
        for (int i = H.groups[g].first; i < H.groups[g].second; ++i) {
          const int64_t numel = matrix_numel(mats[i]);
          add_run(H.in[g], const_cast<void*>(mats[i].grad), mat_io[i].grad_host, grad_bytes(numel, mats[i].grad_dtype));
          if (mat_io[i].param_host)
            add_run(H.out[g], mat_io[i].param_host, mats[i].param_bf16, static_cast<size_t>(numel) * 2);
        }
      for (int i = 0; i < n_vecs; ++i) {
        if (vecs[i].numel == 0) continue;
        add_run(H.a_in, const_cast<void*>(vecs[i].grad), vec_io[i].grad_host,
                grad_bytes(vecs[i].numel, vecs[i].grad_dtype));
        if (vec_io[i].param_host)
          add_run(H.a_out, vec_io[i].param_host, vecs[i].param_bf16, static_cast<size_t>(vecs[i].numel) * 2);
      }
      H.key.swap(key);
    }
  }
  const auto& groups = H.groups;
  const int G = static_cast<int>(groups.size());
  enum { kStart, kAdamIn, kAdamDone, kEndH2d, kEndD2h, kFixed };
  st = ensure_events(ctx, kFixed + 2 * static_cast<size_t>(G));
  if (st != DMUON_OK) return st;
  auto ev = [&](int i) { return ctx->events[static_cast<size_t>(i)]; };
  auto ev_in = [&](int g) { return ev(kFixed + g); };
  auto ev_done = [&](int g) { return ev(kFixed + G + g); };

  // Plans of every group before anything is enqueued: a plan that grows the
  // workspace makes the earlier ones stale, so repeat until all are current.
  const bool fp32 = n_mats > 0 && (muon->flags & DMUON_FLAG_FP32_NS) != 0;
  std::vector<MuonSlot*> slot(static_cast<size_t>(G));
  for (int pass = 0; pass < 3; ++pass) {
    bool all_current = true;
    for (int g = 0; g < G; ++g) {
      slot[static_cast<size_t>(g)] = get_slot(ctx, kSlotHost + static_cast<size_t>(g));
      if (!slot[static_cast<size_t>(g)]) return set_error(DMUON_ERR_NOMEM, "step_host: host allocation failed");
      st = prepare_slot(ctx, *slot[static_cast<size_t>(g)], mats + groups[static_cast<size_t>(g)].first,
                        groups[static_cast<size_t>(g)].second - groups[static_cast<size_t>(g)].first, fp32);
      if (st != DMUON_OK) return st;
    }
    for (int g = 0; g < G; ++g) all_current = all_current && slot[static_cast<size_t>(g)]->plan.ws_epoch == ctx->ws_epoch;
    if (all_current) break;
  }

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DM_CUDA(cudaEventRecord(ev(kStart), s));
  DM_CUDA(cudaStreamWaitEvent(ctx->h2d, ev(kStart), 0));
  DM_CUDA(cudaStreamWaitEvent(ctx->d2h, ev(kStart), 0));
  // Whatever happens below, `stream` ends up ordered after both copy streams.
  auto join = [&](int status) {
    if (cudaEventRecord(ev(kEndH2d), ctx->h2d) != cudaSuccess || cudaEventRecord(ev(kEndD2h), ctx->d2h) != cudaSuccess ||
        cudaStreamWaitEvent(s, ev(kEndH2d), 0) != cudaSuccess || cudaStreamWaitEvent(s, ev(kEndD2h), 0) != cudaSuccess) {
      if (status == DMUON_OK) return cuda_fail(cudaGetLastError(), "step_host: joining the copy streams");
    }
    return status;
  };
  // All gradient copies first, in the order the steps consume them.
  for (int g = 0; g < G; ++g) {
    if ((st = enqueue_runs(H.in[static_cast<size_t>(g)], cudaMemcpyHostToDevice, ctx->h2d)) != DMUON_OK) return join(st);
    if (cudaEventRecord(ev_in(g), ctx->h2d) != cudaSuccess) return join(cuda_fail(cudaGetLastError(), "step_host"));
    if (g == 0 && n_vecs > 0) {
      if ((st = enqueue_runs(H.a_in, cudaMemcpyHostToDevice, ctx->h2d)) != DMUON_OK) return join(st);
      if (cudaEventRecord(ev(kAdamIn), ctx->h2d) != cudaSuccess) return join(cuda_fail(cudaGetLastError(), "step_host"));
    }
  }
  if (G == 0 && n_vecs > 0) {
    if ((st = enqueue_runs(H.a_in, cudaMemcpyHostToDevice, ctx->h2d)) != DMUON_OK) return join(st);
    if (cudaEventRecord(ev(kAdamIn), ctx->h2d) != cudaSuccess) return join(cuda_fail(cudaGetLastError(), "step_host"));
  }
  auto adam = [&]() {
    if (cudaStreamWaitEvent(s, ev(kAdamIn), 0) != cudaSuccess) return cuda_fail(cudaGetLastError(), "step_host");
    int r = adamw_step_impl(ctx, vecs, n_vecs, adamw->lr, adamw->beta1, adamw->beta2, adamw->eps, adamw->wd,
                            adamw->step, s);
    if (r != DMUON_OK) return r;
    if (cudaEventRecord(ev(kAdamDone), s) != cudaSuccess || cudaStreamWaitEvent(ctx->d2h, ev(kAdamDone), 0) != cudaSuccess)
      return cuda_fail(cudaGetLastError(), "step_host");
    return enqueue_runs(H.a_out, cudaMemcpyDeviceToHost, ctx->d2h);
  };
  for (int g = 0; g < G; ++g) {
    const int b = groups[static_cast<size_t>(g)].first, e = groups[static_cast<size_t>(g)].second;
    if (cudaStreamWaitEvent(s, ev_in(g), 0) != cudaSuccess) return join(cuda_fail(cudaGetLastError(), "step_host"));
    st = muon_step_impl(ctx, *slot[static_cast<size_t>(g)], mats + b, e - b, muon->lr, muon->momentum, muon->wd,
                        muon->ns_steps, muon->a, muon->b, muon->c, muon->flags, s);
    if (st != DMUON_OK) return join(st);
    if (cudaEventRecord(ev_done(g), s) != cudaSuccess || cudaStreamWaitEvent(ctx->d2h, ev_done(g), 0) != cudaSuccess)
      return join(cuda_fail(cudaGetLastError(), "step_host"));
    if ((st = enqueue_runs(H.out[static_cast<size_t>(g)], cudaMemcpyDeviceToHost, ctx->d2h)) != DMUON_OK) return join(st);
    if (g == 0 && n_vecs > 0 && (st = adam()) != DMUON_OK) return join(st);
  }
  if (G == 0 && n_vecs > 0 && (st = adam()) != DMUON_OK) return join(st);
  return join(DMUON_OK);
}

int dmuon_sync(dmuon_context* ctx, void* stream) {
  clear_error();
  if (!ctx) return set_error(DMUON_ERR_INVALID_ARG, "sync: null context");
  if (!ctx->dev_ready) return DMUON_OK;
  DeviceGuard guard(ctx->device);
  DM_CUDA(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  int word = 0;
  DM_CUDA(cudaMemcpy(&word, ctx->err.p, sizeof(int), cudaMemcpyDeviceToHost));
  if (word != kErrNone) {
    DM_CUDA(cudaMemset(ctx->err.p, 0, sizeof(int)));
    char buf[96];
    snprintf(buf, sizeof buf, "a bounded device-side wait ran out (site %d)", word);
    return set_error(DMUON_ERR_TIMEOUT, buf);
  }
  return DMUON_OK;
}

int dmuon_selftest_wait_timeout(dmuon_context* ctx, int32_t timeout_us, void* stream) {
  clear_error();
  if (!ctx) return set_error(DMUON_ERR_INVALID_ARG, "selftest: null context");
  if (timeout_us < 1 || timeout_us > 2000000)
    return set_error(DMUON_ERR_INVALID_ARG, "selftest: timeout_us outside [1, 2000000]");
  DeviceGuard guard(ctx->device);
  int st = ensure_device(ctx);
  if (st != DMUON_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return timed_launch(ctx, -1, s, [&] {
    return launch_selftest_wait(static_cast<int*>(ctx->err.p), 1000ll * timeout_us, s);
  });
}

int dmuon_profile(dmuon_context* ctx, int32_t enable) {
  clear_error();
  if (!ctx) return set_error(DMUON_ERR_INVALID_ARG, "profile: null context");
  ctx->prof.on = enable != 0;
  return DMUON_OK;
}

int dmuon_profile_read(dmuon_context* ctx, double* ms_out, int64_t* count_out) {
  clear_error();
  if (!ctx || !ms_out) return set_error(DMUON_ERR_INVALID_ARG, "profile_read: null argument");
  Profiler& P = ctx->prof;
  DeviceGuard guard(ctx->device);
  for (auto& p : P.pending) {
    DM_CUDA(cudaEventSynchronize(p.b));
    float ms = 0.f;
    DM_CUDA(cudaEventElapsedTime(&ms, p.a, p.b));
    if (p.kind >= 0 && p.kind < DMUON_KERNEL_KINDS) {
      P.ms[p.kind] += ms;
      P.count[p.kind] += 1;
    }
    P.pool.push_back(p.a);
    P.pool.push_back(p.b);
  }
  P.pending.clear();
  for (int k = 0; k < DMUON_KERNEL_KINDS; ++k) {
    ms_out[k] = P.ms[k];
    if (count_out) count_out[k] = P.count[k];
    P.ms[k] = 0.0;
    P.count[k] = 0;
  }
  return DMUON_OK;
}

int dmuon_set_tuning(int32_t key, int32_t value) {
  clear_error();
  if (key == 1) {
    set_tc_mn_swap(value ? 1 : 0);
    return DMUON_OK;
  }
  if (key == 2) {
    g_ns_pairs = value ? 1 : 0;
    return DMUON_OK;
  }
  if (key == 3) {
    g_tc2_stages_sel = (value == 5) ? 5 : 4;
    set_tc2_variant(g_tc2_stages_sel, g_tc2_prefetch_sel);
    return DMUON_OK;
  }
  if (key == 7) {
    g_fold_diag = value ? 1 : 0;
    return DMUON_OK;
  }
  if (key == 8) {
    if (value < 0 || value > 1000000) return set_error(DMUON_ERR_INVALID_ARG, "set_tuning: key 8 value outside [0, 1e6]");
    g_epi8_below = value;
    return DMUON_OK;
  }
  if (key == 9) {
    if (value < 1 || value > 16) return set_error(DMUON_ERR_INVALID_ARG, "set_tuning: key 9 value outside [1, 16]");
    g_mom_groups = value;
    return DMUON_OK;
  }
  if (key == 10) {
    if (value < 1 || value > 65536) return set_error(DMUON_ERR_INVALID_ARG, "set_tuning: key 10 value outside [1, 65536]");
    g_group_min_elems = int64_t(value) << 20;
    return DMUON_OK;
  }
  if (key == 4) {
    g_tile_order = value ? 1 : 0;
    return DMUON_OK;
  }
  if (key == 6) {
    g_tri = value ? 1 : 0;
    return DMUON_OK;
  }
  if (key == 5) {
    g_tc2_prefetch_sel = value ? 1 : 0;
    set_tc2_variant(g_tc2_stages_sel, g_tc2_prefetch_sel);
    return DMUON_OK;
  }
  return set_error(DMUON_ERR_INVALID_ARG, "set_tuning: unknown key");
}

}  // extern "C"
