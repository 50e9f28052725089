// Launch sequencing of a Muon step over a prepared plan (pointer table,
// momentum and norms, the Newton-Schulz phases, the update), the overlapped
// multi-group step and the AdamW step.
#include "runtime.h"

#include <new>

namespace dmuon {

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
                 size_t ws_base) {
  const std::string key = plan_key(mats, n, fp32, ctx->tune.tile_order);
  if (key == S.plan.key && S.plan.ws_epoch == ctx->ws_epoch && S.plan.ws_base == ws_base) return DMUON_OK;
  int st = build_muon_plan(ctx, S.plan, mats, n, fp32, key, ws_base);
  if (st != DMUON_OK) S.plan.release();
  return st;
}

// Tensors of a bf16 class in plan P (the ones the tensor-core path steps).
std::vector<char> bf16_tensors(const MuonPlan& P, int n) {
  std::vector<char> f(static_cast<size_t>(n), 0);
  for (const SliceRef& R : P.slices)
    if (!P.classes[static_cast<size_t>(R.cls)].f32) f[static_cast<size_t>(R.mat)] = 1;
  return f;
}

// A TMA copy needs a 16-byte-aligned base and rows whose byte length is a
// multiple of 16: n % 4 == 0 for the fp32 master, n % 8 == 0 for the bf16
// parameter.
bool tma_copyable(const dmuon_matrix& M) {
  const int64_t nn = M.shape[M.rank - 1];
  return aligned16(M.master) && nn % 4 == 0 && (!M.param_bf16 || (aligned16(M.param_bf16) && nn % 8 == 0));
}

bool plan_tma_copyable(const MuonPlan& P, const dmuon_matrix* mats, int n) {
  const std::vector<char> f = bf16_tensors(P, n);
  for (int i = 0; i < n; ++i)
    if (f[static_cast<size_t>(i)] && !tma_copyable(mats[i])) return false;
  return true;
}

// Tensor maps of the callers' fp32 masters (32 x 32 boxes) and bf16
// parameters (64 x 32 boxes) for the fused update's TMA copies, per tensor
// of a bf16 class, rebuilt only when the descriptor array or the tensors'
// classes change.  A tensor that is not tma_copyable gets no maps, and then
// no launch of the call fuses the update (the last Combine stores X and the
// streaming pass updates W).
int build_caller_maps(MuonSlot& S, const dmuon_matrix* mats, int n, cudaStream_t s) {
  const MuonPlan& P = S.plan;
  const std::vector<char> bf16_tensor = bf16_tensors(P, n);
  std::vector<uint8_t> key;
  keep_bytes(key, mats, n);
  key.insert(key.end(), bf16_tensor.begin(), bf16_tensor.end());
  if (key == S.cmaps_key && !S.cmaps_host.empty()) return DMUON_OK;
  S.cmaps_host.clear();
  S.map_w.assign(static_cast<size_t>(n), -1);
  S.map_p.assign(static_cast<size_t>(n), -1);
  S.all_tma = true;
  EncodeTiledFn enc = get_encode_fn();
  for (int i = 0; i < n; ++i) {
    if (!bf16_tensor[static_cast<size_t>(i)]) continue;
    const dmuon_matrix& M = mats[i];
    const int64_t m = M.shape[M.rank - 2], nn = M.shape[M.rank - 1];
    int64_t lead = 1;
    for (int d = 0; d < M.rank - 2; ++d) lead *= M.shape[d];
    if (!enc || !tma_copyable(M)) {
      S.all_tma = false;
      continue;
    }
    cuuint64_t dims[3] = {(cuuint64_t)nn, (cuuint64_t)m, (cuuint64_t)lead};
    cuuint32_t estr[3] = {1, 1, 1};
    CUtensorMap mw;
    cuuint64_t sw[2] = {(cuuint64_t)(nn * 4), (cuuint64_t)(m * nn * 4)};
    cuuint32_t bw[3] = {32, 32, 1};
    if (enc(&mw, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, M.master, dims, sw, bw, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
        CUDA_SUCCESS) {
      S.all_tma = false;
      continue;
    }
    S.map_w[static_cast<size_t>(i)] = static_cast<int32_t>(S.cmaps_host.size());
    S.cmaps_host.push_back(mw);
    if (M.param_bf16) {
      CUtensorMap mp;
      cuuint64_t spr[2] = {(cuuint64_t)(nn * 2), (cuuint64_t)(m * nn * 2)};
      cuuint32_t bp[3] = {64, 32, 1};
      if (enc(&mp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, M.param_bf16, dims, spr, bp, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
        S.map_w[static_cast<size_t>(i)] = -1;
        S.cmaps_host.pop_back();
        S.all_tma = false;
        continue;
      }
      S.map_p[static_cast<size_t>(i)] = static_cast<int32_t>(S.cmaps_host.size());
      S.cmaps_host.push_back(mp);
    }
  }
  if (S.cmaps_host.empty()) S.cmaps_host.resize(1);  // keep a valid (unused) table
  int st = S.cmaps.put(S.cmaps_host.data(), S.cmaps_host.size() * sizeof(CUtensorMap), s);
  if (st != DMUON_OK) return st;
  S.cmaps_key.swap(key);
  return DMUON_OK;
}

// Stage 1 of a Muon step on a prepared slot: the per-call pointer table,
// uploaded on stream s.
int muon_stage_table(dmuon_context* ctx, MuonSlot& S, const dmuon_matrix* mats, int n, int32_t ns_steps,
                     cudaStream_t s) {
  int st = check_matrices_reachable(ctx, S.checked, mats, n);
  if (st != DMUON_OK) return st;
  st = build_caller_maps(S, mats, n, s);
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
    D.x0lo = C.f32 ? nullptr : reinterpret_cast<uint16_t*>(ws + C.off_xl) + static_cast<size_t>(R.z) * C.m * C.ld;
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
    D.map_w = S.map_w[static_cast<size_t>(R.mat)];
    D.map_p = S.map_p[static_cast<size_t>(R.mat)];
    D.z_t = static_cast<int32_t>(R.elem_offset / (static_cast<int64_t>(C.m) * C.n));
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
                   float c, cudaStream_t s, bool call_tma) {
  MuonPlan& P = S.plan;
  const SliceDesc* d_slices = static_cast<const SliceDesc*>(S.table.dev.p);
  const Chunk* d_chunks = static_cast<const Chunk*>(P.chunks_dev.p);
  float* inv_norm = static_cast<float*>(P.inv_norm.p);
  const int n_chunks = static_cast<int>(P.chunks.size());
  int st = DMUON_OK;
  // The last Combine applies the update in its epilogue when every tensor
  // of the call has TMA maps (call_tma: the same decision for every group
  // of a grouped call, so grouping never changes a result).  On the CTA-pair
  // kernel (W in, W' and the parameter out by TMA tile copies) that pays at
  // any main-loop length: GPT-2 set 1.90 -> 1.85 ms, many-small set 43.3 ->
  // 42.7 ms per step against a plain X store by 8 epilogue warps plus the
  // streaming update pass.  (The one-CTA kernel's fused epilogue moves W
  // row by row and is slower than the separate pass on short main loops,
  // GPT-2 set 380 against 120 + ~160 us, but a rule that looked at the
  // call's main-loop lengths would differ between the groups of a grouped
  // call.)
  const Tuning& tu = ctx->tune;
  const bool pairs = tu.ns_pairs != 0;
  const bool fuse_last = call_tma && S.all_tma;
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
        if (tu.fold_diag && it >= 2) {
          // X' = a X + B X = (a I + B) X: the Poly adds a on B's diagonal and
          // the Combine reads no aux.
          if (kind == kPoly) T.diag = a;
          if (kind == kCombine) T.a = 0.f;
        }
        if (kind == kCombine && it == ns_steps - 1 && fuse_last) {
          // The last Combine applies the update itself (no X store, no update pass).
          T.fuse_update = 1;
          T.slices = d_slices;
          T.cmaps = static_cast<const CUtensorMap*>(S.cmaps.dev.p);
          T.lr = lr;
          T.wd = wd;
        }
        T.tri = (pairs && tu.tri) ? 1 : 0;
        T.stages = tu.tc2_stages;
        // 256 x 512 tiles where the main loops are long enough to pay for an
        // accumulator that is not double-buffered.
        T.wide = (T.tri && !T.fuse_update && tu.wide_min_kb > 0 && P.phase2w[kind].n_tiles > 0 &&
                  P.phase2[kind].mean_kblocks >= static_cast<double>(tu.wide_min_kb))
                     ? 1
                     : 0;
        const PhaseTiles& PT = pairs ? (T.wide ? P.phase2w[kind] : P.phase2[kind]) : P.phase[kind];
        T.epi8 = (!T.fuse_update && PT.mean_kblocks < static_cast<double>(tu.epi8_below)) ? 1 : 0;
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
  // With a fused last Combine the update pass covers the fp32 classes only;
  // otherwise (or with no iterations) every slice.
  const bool every = ns_steps == 0 || !fuse_last;
  const int n_upd = every ? n_chunks : static_cast<int>(P.chunks_f32.size());
  if (n_upd == 0) return DMUON_OK;
  const Chunk* d_upd = every ? d_chunks : static_cast<const Chunk*>(P.chunks_f32_dev.p);
  return timed_launch(ctx, DMUON_KERNEL_UPDATE, s, [&] {
    return launch_update(d_slices, d_upd, n_upd, lr, wd, 0, ns_steps == 0 ? inv_norm : nullptr, s);
  });
}

// One Muon step of a validated, non-empty tensor list on the current device,
// every stage on stream s.
int muon_step_impl(dmuon_context* ctx, MuonSlot& S, const dmuon_matrix* mats, int n, float lr,
                   float momentum, float wd, int32_t ns_steps, float a, float b, float c,
                   uint32_t flags, cudaStream_t s, bool call_tma) {
  int st = prepare_slot(ctx, S, mats, n, (flags & DMUON_FLAG_FP32_NS) != 0);
  if (st != DMUON_OK) return st;
  st = muon_stage_table(ctx, S, mats, n, ns_steps, s);
  if (st != DMUON_OK) return st;
  st = muon_launch_front(ctx, S, momentum, flags, s);
  if (st != DMUON_OK) return st;
  return muon_launch_ns(ctx, S, lr, wd, ns_steps, a, b, c, s, call_tma);
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
  // Caller's stream: each group's Newton-Schulz once its momentum is done;
  // the update fuses in every group or in none.
  bool call_tma = true;
  for (int g = 0; g < G; ++g) call_tma = call_tma && S[static_cast<size_t>(g)]->all_tma;
  for (int g = 0; g < G; ++g) {
    DM_CUDA(cudaStreamWaitEvent(s, ctx->side_events[2 + static_cast<size_t>(g)], 0));
    st = muon_launch_ns(ctx, *S[static_cast<size_t>(g)], lr, wd, ns_steps, a, b, c, s, call_tma);
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


}  // namespace dmuon
