// The host-buffer step (dmuon_step_host): gradients copied in from
// page-locked host memory and parameters copied out, group by group, on two
// copy streams of the context, overlapped with the other groups' compute.
#include "runtime.h"

namespace dmuon {
namespace {

// Tensor count above which the host-buffer step uses equal group shares.
constexpr int kShapedMaxTensors = 512;

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

// Consecutive groups by Newton-Schulz work (element count when there are no
// iterations), every group non-empty; the shares are set below.
std::vector<std::pair<int, int>> split_groups(const dmuon_matrix* mats, int n, int groups, int ns_steps) {
  std::vector<double> cost(static_cast<size_t>(n));
  double total = 0.0;
  for (int i = 0; i < n; ++i) {
    const dmuon_matrix& M = mats[i];
    const double m = double(M.shape[M.rank - 2]), q0 = double(M.shape[M.rank - 1]);
    const double p = std::min(m, q0), q = std::max(m, q0);
    const double lead = double(matrix_elems(M)) / (m * q0);
    cost[static_cast<size_t>(i)] = ns_steps > 0 ? lead * (4.0 * p * p * q + 2.0 * p * p * p) : lead * m * q0;
    total += cost[static_cast<size_t>(i)];
  }
  // Shares grow from both ends, 2^min(g, G-1-g, 3): the first group's
  // gradients (copied before any compute) and the last group's parameters
  // (copied after all compute) are small, the middle groups large and few.
  // With many tensors the copies' fixed cost (several microseconds each)
  // dominates instead, and equal groups spread it evenly over the step.
  const bool shaped = n <= kShapedMaxTensors;
  std::vector<double> share(static_cast<size_t>(groups));
  double wsum = 0.0;
  for (int g = 0; g < groups; ++g) {
    share[static_cast<size_t>(g)] = shaped ? double(1 << std::min(std::min(g, groups - 1 - g), 3)) : 1.0;
    wsum += share[static_cast<size_t>(g)];
  }
  std::vector<std::pair<int, int>> out;
  int start = 0;
  double acc = 0.0, cum = share[0];  // shares of the groups up to the open one
  for (int i = 0; i < n; ++i) {
    acc += cost[static_cast<size_t>(i)];
    const int closed = static_cast<int>(out.size());
    if (closed < groups - 1 && i + 1 < n && acc >= total * cum / wsum) {
      out.push_back({start, i + 1});
      start = i + 1;
      cum += share[static_cast<size_t>(closed + 1)];
    }
  }
  if (start < n) out.push_back({start, n});
  return out;
}

}  // namespace
}  // namespace dmuon

using namespace dmuon;

extern "C" {

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
  st = check_no_overlap_cached(ctx, mats, n_mats, vecs, n_vecs);
  if (st != DMUON_OK) return st;
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
      // Groups of fewer than host_group_min_elems elements leave their
      // launches too few tiles to fill the GPU (a GPT-2-sized list in 16
      // groups ran twice as long as in 2), so short lists get fewer groups.
      int64_t elems = 0;
      for (int i = 0; i < n_mats; ++i) elems += matrix_elems(mats[i]);
      const int groups =
          static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(n_groups, elems / ctx->tune.host_group_min_elems)));
      H.groups = split_groups(mats, n_mats, groups, n_mats > 0 ? muon->ns_steps : 0);
      const size_t G = H.groups.size();
      H.in.resize(G);
      H.out.resize(G);
      auto grad_bytes = [](int64_t numel, int32_t dtype) {
        return static_cast<size_t>(numel) * (dtype == DMUON_DTYPE_BF16 ? 2 : 4);
      };
      for (size_t g = 0; g < G; ++g)
        for (int i = H.groups[g].first; i < H.groups[g].second; ++i) {
          const int64_t numel = matrix_elems(mats[i]);
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
  enum { kStart, kAdamIn, kAdamDone, kEndH2d, kEndD2h, kH2dAll, kFixed };
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
  // Timeline (profiling only): timing events beside the ordering events.
  const bool tl = ctx->prof.on;
  if (tl) {
    ctx->tl_groups = -1;
    while (ctx->tl_events.size() < 3 + 3 * static_cast<size_t>(G)) {
      cudaEvent_t e = nullptr;
      DM_CUDA(cudaEventCreate(&e));
      ctx->tl_events.push_back(e);
    }
  }
  auto mark = [&](size_t i, cudaStream_t on) {
    if (tl) cudaEventRecord(ctx->tl_events[i], on);
  };
  DM_CUDA(cudaEventRecord(ev(kStart), s));
  mark(0, s);
  DM_CUDA(cudaStreamWaitEvent(ctx->h2d, ev(kStart), 0));
  DM_CUDA(cudaStreamWaitEvent(ctx->d2h, ev(kStart), 0));
  // Whatever happens below, `stream` ends up ordered after both copy streams.
  auto join = [&](int status) {
    mark(2, ctx->d2h);
    if (tl && status == DMUON_OK) ctx->tl_groups = G;
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
    mark(3 + 3 * static_cast<size_t>(g), ctx->h2d);
    if (g == 0 && n_vecs > 0) {
      if ((st = enqueue_runs(H.a_in, cudaMemcpyHostToDevice, ctx->h2d)) != DMUON_OK) return join(st);
      if (cudaEventRecord(ev(kAdamIn), ctx->h2d) != cudaSuccess) return join(cuda_fail(cudaGetLastError(), "step_host"));
    }
  }
  if (G == 0 && n_vecs > 0) {
    if ((st = enqueue_runs(H.a_in, cudaMemcpyHostToDevice, ctx->h2d)) != DMUON_OK) return join(st);
    if (cudaEventRecord(ev(kAdamIn), ctx->h2d) != cudaSuccess) return join(cuda_fail(cudaGetLastError(), "step_host"));
  }
  // Parameter copies start only once every gradient copy has landed.  Where
  // the host link's two directions share one bottleneck (measured: 54 GB/s
  // host to device alone, 92 GB/s for both directions together on one box),
  // early parameter copies would slow the gradient copies that the later
  // groups' compute is waiting for; where they do not, the early groups'
  // parameter copies are not on the critical path anyway.
  // (The timeline's "all gradients in" mark goes here too, right behind the
  // last gradient copy: recorded later, on an idle stream, it would carry
  // the time the host finished enqueueing instead.)
  mark(1, ctx->h2d);
  if (cudaEventRecord(ev(kH2dAll), ctx->h2d) != cudaSuccess || cudaStreamWaitEvent(ctx->d2h, ev(kH2dAll), 0) != cudaSuccess)
    return join(cuda_fail(cudaGetLastError(), "step_host"));
  auto adam = [&]() {
    if (cudaStreamWaitEvent(s, ev(kAdamIn), 0) != cudaSuccess) return cuda_fail(cudaGetLastError(), "step_host");
    int r = adamw_step_impl(ctx, vecs, n_vecs, adamw->lr, adamw->beta1, adamw->beta2, adamw->eps, adamw->wd,
                            adamw->step, s);
    if (r != DMUON_OK) return r;
    if (cudaEventRecord(ev(kAdamDone), s) != cudaSuccess || cudaStreamWaitEvent(ctx->d2h, ev(kAdamDone), 0) != cudaSuccess)
      return cuda_fail(cudaGetLastError(), "step_host");
    return enqueue_runs(H.a_out, cudaMemcpyDeviceToHost, ctx->d2h);
  };
  // The update fuses in every group or in none, as in one dmuon_muon_step
  // over all tensors, so the grouping never changes a result.
  bool call_tma = true;
  for (int g = 0; g < G; ++g) {
    const int b = groups[static_cast<size_t>(g)].first, e = groups[static_cast<size_t>(g)].second;
    call_tma = call_tma && plan_tma_copyable(slot[static_cast<size_t>(g)]->plan, mats + b, e - b);
  }
  for (int g = 0; g < G; ++g) {
    const int b = groups[static_cast<size_t>(g)].first, e = groups[static_cast<size_t>(g)].second;
    if (cudaStreamWaitEvent(s, ev_in(g), 0) != cudaSuccess) return join(cuda_fail(cudaGetLastError(), "step_host"));
    st = muon_step_impl(ctx, *slot[static_cast<size_t>(g)], mats + b, e - b, muon->lr, muon->momentum, muon->wd,
                        muon->ns_steps, muon->a, muon->b, muon->c, muon->flags, s, call_tma);
    if (st != DMUON_OK) return join(st);
    if (cudaEventRecord(ev_done(g), s) != cudaSuccess || cudaStreamWaitEvent(ctx->d2h, ev_done(g), 0) != cudaSuccess)
      return join(cuda_fail(cudaGetLastError(), "step_host"));
    mark(4 + 3 * static_cast<size_t>(g), s);
    if ((st = enqueue_runs(H.out[static_cast<size_t>(g)], cudaMemcpyDeviceToHost, ctx->d2h)) != DMUON_OK) return join(st);
    mark(5 + 3 * static_cast<size_t>(g), ctx->d2h);
    if (g == 0 && n_vecs > 0 && (st = adam()) != DMUON_OK) return join(st);
  }
  if (G == 0 && n_vecs > 0 && (st = adam()) != DMUON_OK) return join(st);
  return join(DMUON_OK);
}

int dmuon_profile_host_timeline(dmuon_context* ctx, double* ms_out, int32_t capacity, int32_t* n_groups_out) {
  clear_error();
  if (!ctx || !ms_out || !n_groups_out || capacity < 0)
    return set_error(DMUON_ERR_INVALID_ARG, "profile_host_timeline: null argument or negative capacity");
  *n_groups_out = 0;
  if (ctx->tl_groups < 0) return DMUON_OK;
  const int G = ctx->tl_groups;
  *n_groups_out = G;
  if (capacity < 2 + 3 * G) return set_error(DMUON_ERR_INVALID_ARG, "profile_host_timeline: capacity < 2 + 3 * groups");
  DeviceGuard guard(ctx->device);
  auto at = [&](size_t i, double* out) -> int {
    DM_CUDA(cudaEventSynchronize(ctx->tl_events[i]));
    float ms = 0.f;
    DM_CUDA(cudaEventElapsedTime(&ms, ctx->tl_events[0], ctx->tl_events[i]));
    *out = ms;
    return DMUON_OK;
  };
  int st;
  if ((st = at(1, &ms_out[0])) != DMUON_OK || (st = at(2, &ms_out[1])) != DMUON_OK) return st;
  for (int g = 0; g < G; ++g)
    for (int k = 0; k < 3; ++k)
      if ((st = at(3 + 3 * static_cast<size_t>(g) + static_cast<size_t>(k), &ms_out[2 + 3 * g + k])) != DMUON_OK)
        return st;
  return DMUON_OK;
}

}  // extern "C"
