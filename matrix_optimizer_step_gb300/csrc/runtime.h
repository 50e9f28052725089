// Private runtime of the C ABI, shared by its translation units (api.cu,
// plan.cu, step.cu, host_io.cu): device buffers, plans, the context, and
// the planning and launch-sequencing functions.  Not part of the public ABI
// (include/dmuon.h is).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <memory>
#include <string>
#include <utility>
#include <vector>

#include "../../include/dmuon.h"
#include "host_util.h"
#include "internal.h"

namespace dmuon {

// Kernel and planning policy of a context (dmuon_context_set_tuning).  A new
// context copies the process-wide defaults (dmuon_set_tuning, api.cu).
struct Tuning {
  // Which tensor-core kernel runs the NS phases: 1 = CTA pairs on 256 x 256
  // tiles, 0 = one CTA per 128 x 256 tile.
  int ns_pairs = 1;
  // Tile order inside one problem: 1 = longer tile dimension outer, 0 = rows outer.
  int tile_order = 1;
  // CTA-pair kernel: 1 = symmetric outputs stored as upper blocks only and
  // read through transposed loads, 0 = mirrored stores.
  int tri = 1;
  // Ring depth of the CTA-pair kernel (4 or 5).
  int tc2_stages = 4;
  // From the third iteration on (where X is read back in bf16 anyway), fold
  // the a*X term of the Combine into the Poly output: B + a I.  1 = on.
  int fold_diag = 1;
  // CTA-pair kernel: launches whose tiles average fewer 64-deep k-blocks
  // than this drain their accumulators with 8 epilogue warps instead of 4,
  // and a last Combine that short is not fused with the update.
  int epi8_below = 32;
  // CTA-pair kernel: launches whose tiles average at least this many
  // k-blocks use 256 x 512 tiles where two column blocks fit (0 = never).
  // Measured on the Llama-3-8B and MoE sets: the Gram launches (mean 157
  // and 224 k-blocks) gain 3-6 %.
  int wide_min_kb = 128;
  // Momentum overlapped with Newton-Schulz: a large tensor list is cut into
  // this many groups with disjoint workspace regions, and group g+1's
  // momentum pass (HBM-bound) runs on a side stream while group g's
  // Newton-Schulz products (tensor-core-bound) run on the caller's stream.
  // 1 = one group, everything on the caller's stream.  A group gets at
  // least group_min_elems elements: smaller groups leave their launches too
  // few tiles to fill the GPU, which costs more than the hidden momentum
  // pass saves (measured: a GPT-2-sized list in 4 groups runs 40 % slower,
  // the Llama-3-8B set 1 % faster).  Off by default: the gain is small, and
  // kernels sharing the GPU make per-kernel timings (and the rooflines
  // computed from them) describe the contention rather than the kernels.
  int mom_groups = 1;
  int64_t group_min_elems = int64_t(1) << 30;
  // Host-buffer step: smallest group (elements).
  int64_t host_group_min_elems = int64_t(1) << 25;
};

// Apply one (key, value) pair of dmuon_set_tuning to `t`; DMUON_ERR_INVALID_ARG
// for an unknown key or a value out of range (api.cu).
int apply_tuning(Tuning& t, int32_t key, int32_t value);

// Plan slots of a context: 0 = one-group step, 1.. = overlapped momentum
// groups, 65.. = host-pipeline groups.
constexpr size_t kSlotOverlap = 1, kSlotHost = 65;

int cuda_fail(cudaError_t e, const char* where);

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

using PointerAttrFn = CUresult (*)(void*, CUpointer_attribute, CUdeviceptr);
EncodeTiledFn get_encode_fn();
PointerAttrFn get_pointer_attr_fn();

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

int dev_alloc(DevBuf& b, size_t bytes);

template <class T>
inline int upload(DevBuf& b, const std::vector<T>& v) {
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
  size_t off_xl, off_al;          // low bf16 halves of X and A (bf16 classes only)
  int32_t map_xk[2], map_xmn[2], map_a, map_b, map_a_mn, map_b_mn;
  int32_t map_x_st[2], map_a_st, map_b_st;  // 64 x 32 boxes for TMA stores
  int32_t map_xl_st, map_al_st;              // the same for the low halves
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
  PhaseTiles phase2w[3];    // CTA-pair tiles with 256 x 512 tiles where they fit
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
    for (auto* ph : {phase, phase2, phase2w, phase_f32})
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
  // Tensor maps of the callers' masters and parameters for the fused
  // update's TMA stores, rebuilt when the descriptor array changes.
  StagedTable cmaps;
  std::vector<uint8_t> cmaps_key;
  std::vector<CUtensorMap> cmaps_host;
  std::vector<int32_t> map_w, map_p;  // per tensor of the call, -1 = not storable by TMA
  bool all_tma = false;               // every bf16-class tensor has its maps
  void release() {
    plan.release();
    table.release();
    checked.clear();
    cmaps.release();
    cmaps_key.clear();
    cmaps_host.clear();
    map_w.clear();
    map_p.clear();
    all_tma = false;
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
  dmuon::Tuning tune;
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
  // Descriptor arrays (Muon, AdamW) that last passed the overlap check.
  std::vector<uint8_t> checked_overlap;
  // Host pipeline: copy streams, events, cached groups and copy lists.
  cudaStream_t h2d = nullptr, d2h = nullptr;
  std::vector<cudaEvent_t> events;
  dmuon::HostPlan host;
  // Overlapped momentum: side stream and its events.
  cudaStream_t side = nullptr;
  std::vector<cudaEvent_t> side_events;
  // Timeline of the last host-buffer step made while profiling: timing
  // events at the start, the end of all gradient copies, the end of all
  // copies, and per group the end of its gradient copies, of its compute and
  // of its parameter copies.  tl_groups < 0: none recorded.
  std::vector<cudaEvent_t> tl_events;
  int tl_groups = -1;
};

namespace dmuon {

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

inline bool finite(float x) { return std::isfinite(x); }

inline int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <class T>
inline bool same_bytes(const std::vector<uint8_t>& v, const T* a, int n) {
  return v.size() == sizeof(T) * static_cast<size_t>(n) && memcmp(v.data(), a, v.size()) == 0;
}

template <class T>
inline void keep_bytes(std::vector<uint8_t>& v, const T* a, int n) {
  v.assign(reinterpret_cast<const uint8_t*>(a), reinterpret_cast<const uint8_t*>(a) + sizeof(T) * static_cast<size_t>(n));
}

// ---- api.cu
int ensure_device(dmuon_context* ctx);
int check_matrices_reachable(dmuon_context* ctx, std::vector<uint8_t>& checked, const dmuon_matrix* mats,
                             int n);
int check_vectors_reachable(dmuon_context* ctx, const dmuon_vector* ts, int n);
int check_no_overlap_cached(dmuon_context* ctx, const dmuon_matrix* mats, int n, const dmuon_vector* vecs, int nv);
int validate_muon_call(const dmuon_matrix* mats, int32_t n, float lr, float momentum, float wd,
                       int32_t ns_steps, float a, float b, float c, uint32_t flags);
int validate_adamw_call(const dmuon_vector* ts, int32_t n, float lr, float beta1, float beta2, float eps,
                        float wd, int64_t step);

// ---- plan.cu
std::string plan_key(const dmuon_matrix* mats, int n, bool fp32, int tile_order);
int layout_plan(MuonPlan& P, const dmuon_matrix* mats, int n, bool fp32, size_t ws_base);
size_t plan_ws_bytes(const dmuon_matrix* mats, int n, bool fp32);
int ensure_workspace(dmuon_context* ctx, size_t bytes);
int build_muon_plan(dmuon_context* ctx, MuonPlan& P, const dmuon_matrix* mats, int n, bool fp32,
                    const std::string& key, size_t ws_base);

// ---- step.cu
MuonSlot* get_slot(dmuon_context* ctx, size_t i);
int prepare_slot(dmuon_context* ctx, MuonSlot& S, const dmuon_matrix* mats, int n, bool fp32,
                 size_t ws_base = 0);
int muon_stage_table(dmuon_context* ctx, MuonSlot& S, const dmuon_matrix* mats, int n, int32_t ns_steps,
                     cudaStream_t s);
int muon_launch_front(dmuon_context* ctx, MuonSlot& S, float momentum, uint32_t flags, cudaStream_t s);
// call_tma: every tensor of the whole call (all groups of a grouped call)
// can take the fused update's TMA copies; false keeps every group unfused.
int muon_launch_ns(dmuon_context* ctx, MuonSlot& S, float lr, float wd, int32_t ns_steps, float a, float b,
                   float c, cudaStream_t s, bool call_tma = true);
int muon_step_impl(dmuon_context* ctx, MuonSlot& S, const dmuon_matrix* mats, int n, float lr,
                   float momentum, float wd, int32_t ns_steps, float a, float b, float c,
                   uint32_t flags, cudaStream_t s, bool call_tma = true);
// Whether every bf16-class tensor of plan P (over mats[0..n)) can take the
// fused update's TMA copies.
bool plan_tma_copyable(const MuonPlan& P, const dmuon_matrix* mats, int n);
int64_t matrix_elems(const dmuon_matrix& M);
int muon_step_overlapped(dmuon_context* ctx, const dmuon_matrix* mats, int n, int groups, float lr,
                         float momentum, float wd, int32_t ns_steps, float a, float b, float c,
                         uint32_t flags, cudaStream_t s);
int adamw_step_impl(dmuon_context* ctx, const dmuon_vector* ts, int n, float lr, float beta1, float beta2,
                    float eps, float wd, int64_t step, cudaStream_t s);

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

}  // namespace dmuon
