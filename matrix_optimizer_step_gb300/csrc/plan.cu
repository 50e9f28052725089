// Planning of a Muon step: slices, shape classes, workspace layout, TMA
// tensor maps, problem tables and the balanced tile lists of every phase.
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
#include "runtime.h"

namespace dmuon {

std::string plan_key(const dmuon_matrix* mats, int n, bool fp32, int tile_order) {
  std::string k = fp32 ? "f32|" : "bf16|";
  k += "o" + std::to_string(tile_order) + "|";
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
// 2 = CTA-pair tcgen05 tiles, 3 = CTA-pair tiles where two adjacent column
// blocks of one row block form a 256 x 512 tile (kTileWideBit) wherever both
// exist (for a symmetric output: both on or above the diagonal).
// `slots` = persistent CTAs (or CTA pairs).
int build_phase_tiles(const std::vector<NsProblem>& probs, int geometry, int slots, int tile_order,
                      PhaseTiles& out) {
  const bool fp32 = geometry == 0;
  const bool wide = geometry == 3;
  const int bm = geometry == 0 ? kSimtBM : geometry == 1 ? kTcBM : kTc2Tile;
  const int bn = geometry == 0 ? kSimtBN : geometry == 1 ? kTcBN : kTc2Tile;
  std::vector<uint2> tiles;
  std::vector<int64_t> cost;
  double kb_sum = 0.0;
  for (size_t p = 0; p < probs.size(); ++p) {
    const NsProblem& P = probs[p];
    const int tm = (P.M + bm - 1) / bm, tn = (P.N + bn - 1) / bn;
    if (tm > 0xFFFF || tn > 0xFFFF) return set_error(DMUON_ERR_SHAPE, "matrix too large for the tile index");
    const int64_t kb = (P.K + kTcBK - 1) / kTcBK;
    // A wide tile moves 1.5x the operand bytes of a narrow one per k-block.
    const int64_t c = kb + 2, c_wide = kb + kb / 2 + 3;
    auto add = [&](int i, int j, bool w) {
      const uint32_t x = static_cast<uint32_t>(p) | (w ? kTileWideBit : 0u);
      tiles.push_back(make_uint2(x, (static_cast<uint32_t>(i) << 16) | static_cast<uint32_t>(j)));
      cost.push_back(w ? c_wide : c);
      kb_sum += static_cast<double>(kb);
    };
    // Tiles of equal cost run in list order, so consecutive tiles run at the
    // same time: walk the longer tile dimension in the outer loop, so a wave
    // shares few panels of the larger operand (which then stay in L2).
    const bool n_outer = tile_order && tn > tm;
    const int jstep = wide ? 2 : 1;
    if (n_outer) {
      for (int j = 0; j < tn; j += jstep)
        for (int i = 0; i < tm; ++i) {
          if (P.sym && (i * bm) / bn > j) continue;  // below the diagonal: mirrored
          add(i, j, wide && j + 1 < tn);
        }
    } else {
      for (int i = 0; i < tm; ++i) {
        const int j0 = P.sym ? (i * bm) / bn : 0;  // first block on or above the diagonal
        for (int j = j0; j < tn; j += (wide && j + 1 < tn) ? 2 : 1) add(i, j, wide && j + 1 < tn);
      }
    }
  }
  out.n_tiles = static_cast<int32_t>(tiles.size());
  out.mean_kblocks = tiles.empty() ? 0.0 : kb_sum / static_cast<double>(tiles.size());
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
    C.off_xl = C.f32 ? 0 : take(static_cast<size_t>(C.count) * C.m * C.ld * 2);
    C.off_al = C.f32 ? 0 : take(static_cast<size_t>(C.count) * p * C.ldp * 2);
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
      st = make_map(enc, &st_map, ws + C.off_xl, C.n, C.m, C.count, C.ld, 64, 32);
      if (st != DMUON_OK) return st;
      C.map_xl_st = static_cast<int32_t>(maps.size());
      maps.push_back(st_map);
      st = make_map(enc, &st_map, ws + C.off_al, p, p, C.count, C.ldp, 64, 32);
      if (st != DMUON_OK) return st;
      C.map_al_st = static_cast<int32_t>(maps.size());
      maps.push_back(st_map);
    }
    st = upload(P.maps, maps);
    if (st != DMUON_OK) return st;
  }

  // Problems of the three phases.  bf16 classes, variant 0/1: X in buffer
  // 0/1, everything bf16.  Variant 2 (first iteration, X in buffer 0) and 3
  // (second iteration, X in buffer 1) add the low bf16 halves: the first
  // Gram also writes A's low half, the first Poly reads A with it, the first
  // Combine reads X0 with its low half (written by the momentum pass) and
  // writes X1's low half over it (each element is read before it is
  // written, by the same thread), and the second Combine reads X1 with that
  // low half.  fp32 classes (all of them in validation mode) go to separate
  // lists with variants 0/1 only.
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
    uint16_t* Xl = C.f32 ? nullptr : reinterpret_cast<uint16_t*>(ws + C.off_xl) + xoff;
    uint16_t* Al = C.f32 ? nullptr : reinterpret_cast<uint16_t*>(ws + C.off_al) + poff;
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
        g.out_lo = Al;
        g.map_out_lo = C.map_al_st;
        y.aux_lo = Al;
        c.aux_lo = Xl;
        c.out_lo = Xl;  // X1's low half over X0's: each element is read before it is written
        c.map_out_lo = C.map_xl_st;
      }
      if (par == 1) c.aux_lo = Xl;
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
      st = build_phase_tiles(var_f32[kind][0], 0, ctx->num_sms, ctx->tune.tile_order, P.phase_f32[kind]);
      if (st != DMUON_OK) return st;
    }
    if (!var[kind][0].empty()) {
      st = build_phase_tiles(var[kind][0], 1, ctx->num_sms, ctx->tune.tile_order, P.phase[kind]);
      if (st != DMUON_OK) return st;
      const int pairs = std::max(1, std::min(ctx->num_sms / 2, ns_tc2_max_pairs()));
      st = build_phase_tiles(var[kind][0], 2, pairs, ctx->tune.tile_order, P.phase2[kind]);
      if (st != DMUON_OK) return st;
      st = build_phase_tiles(var[kind][0], 3, pairs, ctx->tune.tile_order, P.phase2w[kind]);
      if (st != DMUON_OK) return st;
    }
  }
  P.key = key;
  P.ws_epoch = ctx->ws_epoch;
  return DMUON_OK;
}

}  // namespace dmuon
