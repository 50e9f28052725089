// C ABI of the owner-side Muon / AdamW step: the exported entry points,
// argument validation, device set-up and the tuning switches.  Planning is
// in plan.cu, launch sequencing in step.cu, the host-buffer step in
// host_io.cu; every arithmetic step runs in the kernels (k_stream.cu,
// k_ns_tc2.cu, k_ns_tc.cu, k_ns_simt.cu).
#include "runtime.h"

#include <algorithm>

#include <mutex>
#include <new>

namespace dmuon {


// Defaults copied into every new context (dmuon_set_tuning).
namespace {
std::mutex g_tuning_mu;
Tuning g_tuning_defaults;
}  // namespace

int apply_tuning(Tuning& t, int32_t key, int32_t value) {
  switch (key) {
    case 2: t.ns_pairs = value ? 1 : 0; return DMUON_OK;
    case 3: t.tc2_stages = (value == 5) ? 5 : 4; return DMUON_OK;
    case 4: t.tile_order = value ? 1 : 0; return DMUON_OK;
    case 6: t.tri = value ? 1 : 0; return DMUON_OK;
    case 7: t.fold_diag = value ? 1 : 0; return DMUON_OK;
    case 8:
      if (value < 0 || value > 1000000) return set_error(DMUON_ERR_INVALID_ARG, "set_tuning: key 8 value outside [0, 1e6]");
      t.epi8_below = value;
      return DMUON_OK;
    case 9:
      if (value < 1 || value > 16) return set_error(DMUON_ERR_INVALID_ARG, "set_tuning: key 9 value outside [1, 16]");
      t.mom_groups = value;
      return DMUON_OK;
    case 10:
      if (value < 1 || value > 65536)
        return set_error(DMUON_ERR_INVALID_ARG, "set_tuning: key 10 value outside [1, 65536]");
      t.group_min_elems = int64_t(value) << 20;
      return DMUON_OK;
    case 11:
      if (value < 1 || value > (1 << 20))
        return set_error(DMUON_ERR_INVALID_ARG, "set_tuning: key 11 value outside [1, 2^20]");
      t.host_group_min_elems = int64_t(value) << 10;
      return DMUON_OK;
    case 12:
      if (value < 0 || value > 1000000)
        return set_error(DMUON_ERR_INVALID_ARG, "set_tuning: key 12 value outside [0, 1e6]");
      t.wide_min_kb = value;
      return DMUON_OK;
    default:
      return set_error(DMUON_ERR_INVALID_ARG, "set_tuning: unknown key");
  }
}

// ------------------------------------------------------------------ errors
namespace {
thread_local std::string g_last_error;
}

int set_error(int status, const char* msg) {
  g_last_error = msg ? msg : "";
  return status;
}
void clear_error() { g_last_error.clear(); }

int cuda_fail(cudaError_t e, const char* where) {
  std::string m = std::string(where) + ": " + cudaGetErrorString(e);
  return set_error(DMUON_ERR_CUDA, m.c_str());
}

EncodeTiledFn get_encode_fn() {
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


PointerAttrFn get_pointer_attr_fn() {
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

int dev_alloc(DevBuf& b, size_t bytes) {
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

// Memory the step writes must not be shared: no written range (master,
// momentum, bf16 param; AdamW master and moments) may overlap another
// written range or any gradient, within a tensor or across the tensors of a
// call (two entries writing the same memory race).  Gradients are only read
// and may overlap each other.  Host only: the ranges are sorted by start and
// each gradient is searched among them.
namespace {
struct Span {
  uintptr_t lo, hi;  // [lo, hi)
  int route;         // 0 Muon, 1 AdamW
  int idx;
  const char* what;
};
}  // namespace

int check_no_overlap(const dmuon_matrix* mats, int n, const dmuon_vector* vecs, int nv) {
  std::vector<Span> w, r;
  auto add = [](std::vector<Span>& v, const void* p, int64_t bytes, int route, int idx, const char* what) {
    if (!p || bytes <= 0) return;
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    v.push_back(Span{lo, lo + static_cast<uintptr_t>(bytes), route, idx, what});
  };
  for (int i = 0; i < n; ++i) {
    const dmuon_matrix& M = mats[i];
    int64_t numel = 1;
    for (int d = 0; d < M.rank; ++d) numel *= M.shape[d];
    add(w, M.master, 4 * numel, 0, i, "master");
    add(w, M.momentum, 4 * numel, 0, i, "momentum");
    add(w, M.param_bf16, 2 * numel, 0, i, "param");
    add(r, M.grad, (M.grad_dtype == DMUON_DTYPE_BF16 ? 2 : 4) * numel, 0, i, "grad");
  }
  for (int i = 0; i < nv; ++i) {
    const dmuon_vector& V = vecs[i];
    add(w, V.master, 4 * V.numel, 1, i, "master");
    add(w, V.exp_avg, 4 * V.numel, 1, i, "exp_avg");
    add(w, V.exp_avg_sq, 4 * V.numel, 1, i, "exp_avg_sq");
    add(w, V.param_bf16, 2 * V.numel, 1, i, "param");
    add(r, V.grad, (V.grad_dtype == DMUON_DTYPE_BF16 ? 2 : 4) * V.numel, 1, i, "grad");
  }
  static const char* route_name[2] = {"Muon", "AdamW"};
  auto fail = [&](const Span& a, const Span& b) {
    char buf[200];
    snprintf(buf, sizeof buf, "%s tensor %d: %s overlaps %s tensor %d: %s (memory the step writes must not be shared)",
             route_name[a.route], a.idx, a.what, route_name[b.route], b.idx, b.what);
    return set_error(DMUON_ERR_INVALID_ARG, buf);
  };
  std::sort(w.begin(), w.end(), [](const Span& a, const Span& b) { return a.lo < b.lo; });
  for (size_t k = 1; k < w.size(); ++k)
    if (w[k].lo < w[k - 1].hi) return fail(w[k - 1], w[k]);
  for (const Span& g : r) {
    // The written span with the largest start below g.hi is the only one
    // that can overlap g, since written spans are disjoint and sorted.
    auto it = std::lower_bound(w.begin(), w.end(), g.hi, [](const Span& a, uintptr_t v) { return a.lo < v; });
    if (it != w.begin()) {
      const Span& c = *(it - 1);
      if (c.hi > g.lo) return fail(c, g);
    }
  }
  return DMUON_OK;
}

// The same check, skipped when the descriptor arrays are byte-for-byte the
// ones that passed last time on this context.
int check_no_overlap_cached(dmuon_context* ctx, const dmuon_matrix* mats, int n, const dmuon_vector* vecs, int nv) {
  std::vector<uint8_t> key;
  key.reserve(sizeof(dmuon_matrix) * static_cast<size_t>(n) + sizeof(dmuon_vector) * static_cast<size_t>(nv) + 8);
  const int32_t counts[2] = {n, nv};
  key.insert(key.end(), reinterpret_cast<const uint8_t*>(counts), reinterpret_cast<const uint8_t*>(counts) + 8);
  if (n > 0)
    key.insert(key.end(), reinterpret_cast<const uint8_t*>(mats),
               reinterpret_cast<const uint8_t*>(mats) + sizeof(dmuon_matrix) * static_cast<size_t>(n));
  if (nv > 0)
    key.insert(key.end(), reinterpret_cast<const uint8_t*>(vecs),
               reinterpret_cast<const uint8_t*>(vecs) + sizeof(dmuon_vector) * static_cast<size_t>(nv));
  if (key == ctx->checked_overlap) return DMUON_OK;
  const int st = check_no_overlap(mats, n, vecs, nv);
  if (st == DMUON_OK) ctx->checked_overlap.swap(key);
  return st;
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
  {
    std::lock_guard<std::mutex> lock(g_tuning_mu);
    c->tune = g_tuning_defaults;
  }
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
    for (cudaEvent_t e : ctx->tl_events) cudaEventDestroy(e);
    ctx->tl_events.clear();
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
  st = check_no_overlap_cached(ctx, mats, n, nullptr, 0);
  if (st != DMUON_OK) return st;
  DeviceGuard guard(ctx->device);
  st = ensure_device(ctx);
  if (st != DMUON_OK) return st;
  int64_t total = 0;
  for (int i = 0; i < n; ++i) total += matrix_elems(mats[i]);
  const int groups =
      static_cast<int>(std::min<int64_t>({int64_t(ctx->tune.mom_groups), int64_t(n), total / ctx->tune.group_min_elems}));
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
  st = check_no_overlap_cached(ctx, nullptr, 0, ts, n);
  if (st != DMUON_OK) return st;
  DeviceGuard guard(ctx->device);
  st = ensure_device(ctx);
  if (st != DMUON_OK) return st;
  return adamw_step_impl(ctx, ts, n, lr, beta1, beta2, eps, wd, step, static_cast<cudaStream_t>(stream));
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
  if (timeout_us < 1 || timeout_us > 2000000)
    return set_error(DMUON_ERR_INVALID_ARG, "selftest: timeout_us outside [1, 2000000]");
  if (!ctx) {
    // The allocation-free entry point's error word on the current device.
    int* word = nullptr;
    const int st = noalloc_error_word(&word);
    if (st != DMUON_OK) return st;
    const cudaError_t e = launch_selftest_wait(word, 1000ll * timeout_us, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DMUON_OK : cuda_fail(e, "selftest launch");
  }
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
  std::lock_guard<std::mutex> lock(g_tuning_mu);
  Tuning t = g_tuning_defaults;
  const int st = apply_tuning(t, key, value);
  if (st == DMUON_OK) g_tuning_defaults = t;
  return st;
}

int dmuon_context_set_tuning(dmuon_context* ctx, int32_t key, int32_t value) {
  clear_error();
  if (!ctx) return set_error(DMUON_ERR_INVALID_ARG, "context_set_tuning: null context");
  Tuning t = ctx->tune;
  const int st = apply_tuning(t, key, value);
  if (st == DMUON_OK) ctx->tune = t;
  return st;
}

}  // extern "C"
