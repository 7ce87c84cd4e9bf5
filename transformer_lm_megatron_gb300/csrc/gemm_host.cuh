// Host side of the tcgen05 GEMM: TMA descriptors of the operands and outputs,
// the choice of variant (single CTA or CTA pair), tile order and L2 policy, and the
// launch.  Included by gb_mlp.cu inside its anonymous namespace; it uses that
// file's DeviceState, fail(), g_encode, g_launches, launch_kernel() and
// trace_pre()/trace_post().
#pragma once

// L2 policies of the GEMMs' TMA copies (see k_gemm_bf16_tc): none by default.
std::atomic<int> g_l2_hints{0};

// Bytes of the smaller GEMM operand meant to stay in L2 during a grouped sweep.
constexpr int64_t kGroupBytes = 32ll << 20;

// -1: CTA pairs whenever a tile has more than 128 rows; 0: single CTAs; 1: CTA pairs.
std::atomic<int> g_pair_mode{-1};

// Scheduling choices that change no result, kept switchable to measure them:
// paced epilogue stores, and late dependency waits of mlp_bwd's last GEMMs.
std::atomic<int> g_epi_pace{1};
std::atomic<int> g_late_wait{1};
std::atomic<int> g_split_tail{1};
// Tile order: 1 dynamic (a counter per stream region) for every GEMM, 0 static
// round-robin for every GEMM, -1 (the default) dynamic for the batched attention
// products only.  Measured: on the MT-NLG MLP block the dynamic order changed no
// DRAM traffic and was 2 % slower (its weight-gradient GEMMs 9 %); on the causal
// attention products, whose tiles carry unequal work, it was 4-9 % faster.
std::atomic<int> g_tile_sched{-1};

// Late dependency waits pay only for short GEMMs: there the next launch's tiles
// fill the partial last wave and the pipeline drain of the one before.  Tiles are
// dealt to CTAs statically, so on a GEMM of many waves the CTAs that started early
// only finish early, and the idle time moves to the end of the chain instead of
// going away (measured: slightly slower on the 6.9 TFLOP GEMMs of the MT-NLG
// layer, faster on GEMMs of 0.3 TFLOP and below).
constexpr double kLateWaitMaxFlop = 5.5e11;

// 2-D bf16 tensor map: `inner` contiguous elements per row, `outer` rows, row
// pitch `ld` elements; box {box_inner, box_outer}; 128-byte swizzle; out-of-range
// elements read as zero.
int make_map(CUtensorMap* m, const void* base, int64_t inner, int64_t outer, int64_t ld, uint32_t box_inner,
             uint32_t box_outer) {
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MLP_ECUDA, "cuTensorMapEncodeTiled failed (%d): inner %lld outer %lld ld %lld", (int)r,
                (long long)inner, (long long)outer, (long long)ld);
  return MLP_OK;
}

// 2-D fp32 tensor map of a GEMM output for TMA stores / reduce-adds: box of 32
// columns x 32 rows, 128-byte swizzle.
int make_out_map(CUtensorMap* m, const float* base, int64_t cols, int64_t rows, int64_t ld) {
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 4};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MLP_ECUDA, "cuTensorMapEncodeTiled (fp32 output) failed (%d): cols %lld rows %lld ld %lld", (int)r,
                (long long)cols, (long long)rows, (long long)ld);
  return MLP_OK;
}

// 2-D bf16 tensor map of a GEMM output for TMA stores: box of 32 columns x 32
// rows, 64-byte swizzle.
int make_out_map_bf16(CUtensorMap* m, const uint16_t* base, int64_t cols, int64_t rows, int64_t ld) {
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MLP_ECUDA, "cuTensorMapEncodeTiled (bf16 output) failed (%d): cols %lld rows %lld ld %lld", (int)r,
                (long long)cols, (long long)rows, (long long)ld);
  return MLP_OK;
}

// Tensor map of one GEMM operand with `mn` rows/columns along M (or N) and `k`
// along the reduction.  K-major: k contiguous; MN-major: m (or n) contiguous.
int operand_map(CUtensorMap* m, const void* base, bool mn_major, int64_t mn, int64_t k, int64_t ld,
                uint32_t tile_mn) {
  if (mn_major) return make_map(m, base, mn, k, ld, 64, kBK);
  return make_map(m, base, k, mn, ld, kBK, tile_mn);
}

template <bool AM, bool BM, bool PAIR, bool BATCHED = false, bool WIDE = false>
int launch_gemm_t(DeviceState* st, const CUtensorMap& mA, const CUtensorMap& mB, const CUtensorMap& mC,
                  const CUtensorMap& mO0, const CUtensorMap& mO1, int M, int N, int K, const EpiParams& ep,
                  int raster_n_fast, int group, int l2_hints, cudaStream_t stream, int trace_kind, int batch = 1,
                  int nb_h = 1, int causal = kCausalNone, bool late_wait = false) {
  using Cfg = GemmCfg<PAIR, BATCHED || WIDE>;
  auto kern = k_gemm_bf16_tc<AM, BM, PAIR, BATCHED, WIDE>;
  const int slot = (AM ? 2 : 0) + (BM ? 1 : 0) + (PAIR ? 4 : 0) + (BATCHED ? 8 : 0) + (WIDE ? 16 : 0);
  if (!st->gemm_attr[slot]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::kSmemBytes);
    if (e != cudaSuccess) return fail(MLP_ECUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    if (PAIR) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
      cudaLaunchConfig_t qc = {};
      qc.gridDim = dim3(2 * (unsigned)st->sms, 1, 1);
      qc.blockDim = dim3(Cfg::kThreads, 1, 1);
      qc.dynamicSmemBytes = Cfg::kSmemBytes;
      cudaLaunchAttribute qa[1];
      qa[0].id = cudaLaunchAttributeClusterDimension;
      qa[0].val.clusterDim.x = 2;
      qa[0].val.clusterDim.y = 1;
      qa[0].val.clusterDim.z = 1;
      qc.attrs = qa;
      qc.numAttrs = 1;
      int n = 0;
      e = cudaOccupancyMaxActiveClusters(&n, kern, &qc);
      if (e != cudaSuccess || n <= 0) {
        cudaGetLastError();
        n = st->sms / 2;
      }
      st->max_pairs[slot] = n;
    }
    st->gemm_attr[slot] = true;
  }
  const int64_t tiles = (int64_t)((M + Cfg::kTileM - 1) / Cfg::kTileM) * ((N + kBN - 1) / kBN) * batch;
  EpiParams epx = ep;
  epx.pace = g_epi_pace.load(std::memory_order_relaxed);
  late_wait = late_wait && g_late_wait.load(std::memory_order_relaxed) &&
              2.0 * (double)M * (double)N * (double)K * (double)batch <= kLateWaitMaxFlop;
  // Split tail: when the last wave of tiles fills at most half of the CTAs (pairs),
  // its tiles run as two half-reductions each, so that wave takes half as long.
  // Only for bf16 epilogues of plain GEMMs with a reduction of 16 k-blocks or more,
  // and never in a late-waiting launch: the workspace region is shared by all
  // launches on the stream, which therefore must not overlap while they use it.
  const int units = PAIR ? st->max_pairs[slot] : st->sms;
  epx.split_base = (int)tiles;
  epx.split_ws = nullptr;
  epx.split_flags = nullptr;
  int64_t items = tiles;
  if (!BATCHED && !WIDE && causal == kCausalNone && !epi_f32_out(ep.kind) && !late_wait &&
      g_split_tail.load(std::memory_order_relaxed) && (K + kBK - 1) / kBK >= 16) {
    const int64_t rem = tiles % units;
    const int region = (rem > 0 && 2 * rem <= units && rem * (PAIR ? 2 : 1) * 4 <= kSplitSlots)
                           ? split_region(st, stream) : -1;
    if (region >= 0) {
      epx.split_base = (int)(tiles - rem);
      epx.split_ws = st->split_ws + (size_t)region * kSplitSlots * 2 * kSplitSlotFloats;
      epx.split_flags = st->split_flags + (size_t)region * kSplitSlots;
      items = tiles + rem;
    }
  }
  // Dynamic tile order: the stream's tile counters, unless this launch may overlap
  // the previous kernel on the stream (late wait), or the GEMM is one wave.
  const int units_launched = (int)(items < units ? items : units);
  int* sched = nullptr;
  const int order = g_tile_sched.load(std::memory_order_relaxed);
  if ((order == 1 || (order < 0 && BATCHED)) && !late_wait && items > units_launched) {
    const int region = split_region(st, stream);
    if (region >= 0) sched = st->sched_ctr + 2 * region;
  }
  const int ts = trace_pre(stream);
  cudaError_t e;
  if (PAIR) {
    e = launch_kernel(kern, dim3(2 * (unsigned)units_launched), dim3(Cfg::kThreads), Cfg::kSmemBytes, stream, 2, 1, mA,
                      mB, mC, mO0, mO1, M, N, K, epx, raster_n_fast, group, l2_hints, batch, nb_h, causal,
                      late_wait ? 1 : 0, sched, st->status);
  } else {
    e = launch_kernel(kern, dim3((unsigned)units_launched), dim3(Cfg::kThreads), Cfg::kSmemBytes, stream, 1, 1, mA, mB,
                      mC, mO0, mO1, M, N, K, epx, raster_n_fast, group, l2_hints, batch, nb_h, causal,
                      late_wait ? 1 : 0, sched, st->status);
  }
  trace_post(ts, stream, trace_kind, M, N, K);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return fail(MLP_ECUDA, "GEMM launch: %s", cudaGetErrorString(e));
  return MLP_OK;
}

// D[M, N] = A(M x K) B(K x N) with the given operand layouts and epilogue.
// late_wait: the launch reads nothing the previous kernel on the stream writes
// (see k_gemm_bf16_tc); only mlp_bwd's weight-gradient and input-gradient GEMMs,
// never the first kernel of a call.
int gemm(DeviceState* st, const void* a, bool a_mn, int64_t lda, const void* b, bool b_mn, int64_t ldb, int M, int N,
         int K, const EpiParams& ep, cudaStream_t stream, int trace_kind, bool late_wait = false) {
  const int mode = g_pair_mode.load(std::memory_order_relaxed);
  const bool pair = mode == 1 || (mode < 0 && M > kBM);
  CUtensorMap mA, mB, mC, mO0, mO1;
  int rc = operand_map(&mA, a, a_mn, M, K, lda, kBM);
  if (rc) return rc;
  rc = operand_map(&mB, b, b_mn, N, K, ldb, pair ? GemmCfg<true>::kBLoadN : GemmCfg<false>::kBLoadN);
  if (rc) return rc;
  memset(&mC, 0, sizeof(mC));
  memset(&mO0, 0, sizeof(mO0));
  memset(&mO1, 0, sizeof(mO1));
  if (epi_f32_out(ep.kind)) {
    rc = make_out_map(&mC, ep.g_out, N, M, ep.ld);
    if (rc) return rc;
  } else {
    rc = make_out_map_bf16(&mO0, ep.out0, N, M, ep.ld);
    if (rc) return rc;
    if (ep.in0 != nullptr && (ep.kind == kEpiDGelu || ep.kind == kEpiDropRes || ep.kind == kEpiResAdd)) {
      // the bf16 input (U, R or dO), read by the epilogue through TMA
      rc = make_out_map_bf16(&mO1, ep.in0, N, M, ep.ld);
      if (rc) return rc;
    }
    if (ep.kind == kEpiGelu) {
      rc = make_out_map_bf16(&mO1, ep.out1, N, M, ep.ld);
      if (rc) return rc;
    }
  }
  // Visit tiles so that the operand re-read across the sweep is the smaller one.
  // When the two operands are of similar size (the weight-gradient GEMMs, whose
  // reduction runs over the tokens), sweep the fast dimension in groups whose
  // stripes of the smaller operand fit in L2 together (kGroupBytes); the larger
  // operand is then read ceil(blocks / group) times instead of the smaller one
  // being re-read from HBM for every wave.
  const int raster_n_fast = M > N ? 1 : 0;
  const int64_t small_rows = M < N ? M : N;
  const int64_t big_rows = M < N ? N : M;
  int group = 0;
  if (big_rows <= 8 * small_rows) {
    const int64_t stripe_bytes = (int64_t)K * kBN * 2;  // one 256-row block of an operand
    group = (int)(kGroupBytes / stripe_bytes);
    if (group < 1) group = 1;
  }
  const int l2_hints = g_l2_hints.load(std::memory_order_relaxed);
  // Reductions under 16 k-blocks leave the time in the epilogue: 8 epilogue warps.
  const bool wide = (K + kBK - 1) / kBK < 16;
#define GB_LAUNCH(AM_, BM_)                                                                                        \
  (pair ? (wide ? launch_gemm_t<AM_, BM_, true, false, true>(st, mA, mB, mC, mO0, mO1, M, N, K, ep, raster_n_fast,   \
                                                             group, l2_hints, stream, trace_kind, 1, 1, kCausalNone, \
                                                             late_wait)                                              \
                : launch_gemm_t<AM_, BM_, true, false, false>(st, mA, mB, mC, mO0, mO1, M, N, K, ep, raster_n_fast,  \
                                                              group, l2_hints, stream, trace_kind, 1, 1, kCausalNone,\
                                                              late_wait))                                            \
        : (wide ? launch_gemm_t<AM_, BM_, false, false, true>(st, mA, mB, mC, mO0, mO1, M, N, K, ep, raster_n_fast,  \
                                                              group, l2_hints, stream, trace_kind, 1, 1, kCausalNone,\
                                                              late_wait)                                             \
                : launch_gemm_t<AM_, BM_, false, false, false>(st, mA, mB, mC, mO0, mO1, M, N, K, ep, raster_n_fast, \
                                                               group, l2_hints, stream, trace_kind, 1, 1,            \
                                                               kCausalNone, late_wait)))
  if (!a_mn && b_mn) return GB_LAUNCH(false, true);
  if (!a_mn && !b_mn) return GB_LAUNCH(false, false);
  if (a_mn && b_mn) return GB_LAUNCH(true, true);
#undef GB_LAUNCH
  // (MN, K): only the weight-gradient product dB = Y^T dZ with a transposed copy of
  // dZ (mlp_bwd), which always runs on CTA pairs with a deep enough reduction
  if (a_mn && !b_mn && pair && !wide)
    return launch_gemm_t<true, false, true, false, false>(st, mA, mB, mC, mO0, mO1, M, N, K, ep, raster_n_fast, group,
                                                          l2_hints, stream, trace_kind, 1, 1, kCausalNone, late_wait);
  return fail(MLP_EUNSUPPORTED, "operand layout combination not instantiated");
}


// ---------------------------------------------------------------- batched GEMMs
// One operand of a batched GEMM: matrix (b_h, b_s) of a 4-D layout.  `mn` and `k`
// are the extents along M (or N) and the reduction; `ld` is the element distance
// between consecutive rows of the stored matrix (rows run along K for an
// MN-major operand, along M/N for a K-major one); h_stride / s_stride are the
// element distances between consecutive matrices along the two batch indices.
struct BatchOperand {
  const void* base;
  bool mn_major;
  int64_t mn, k, ld, h_stride, s_stride;
};

// One output of a batched GEMM: `cols` = N, `rows` = M of each matrix.
struct BatchOutput {
  void* base;
  int64_t cols, rows, ld, h_stride, s_stride;
};

int make_map4(CUtensorMap* m, CUtensorMapDataType dt, int esz, const void* base, int64_t inner, int64_t rows,
              int64_t ld, int64_t nb_h, int64_t h_stride, int64_t nb_s, int64_t s_stride, uint32_t box_inner,
              uint32_t box_rows, CUtensorMapSwizzle swizzle, CUtensorMapL2promotion prom) {
  cuuint64_t dims[4] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)nb_h, (cuuint64_t)nb_s};
  cuuint64_t strides[3] = {(cuuint64_t)(ld * esz), (cuuint64_t)(h_stride * esz), (cuuint64_t)(s_stride * esz)};
  cuuint32_t box[4] = {box_inner, box_rows, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(m, dt, 4, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle, prom, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MLP_ECUDA, "cuTensorMapEncodeTiled (4-D) failed (%d): inner %lld rows %lld ld %lld strides %lld %lld",
                (int)r, (long long)inner, (long long)rows, (long long)ld, (long long)h_stride, (long long)s_stride);
  return MLP_OK;
}

// nb_h x nb_s independent GEMMs D_b = A_b B_b (M x N, reduction K) with a
// TMA-only epilogue (kEpiStore: bf16 output; kEpiF32Store / kEpiScaleMask: fp32).
int gemm_batched(DeviceState* st, const BatchOperand& a, const BatchOperand& b, const BatchOutput& out, int M, int N,
                 int K, int nb_h, int nb_s, const EpiParams& ep, cudaStream_t stream, int trace_kind,
                 int causal = kCausalNone) {
  if ((!epi_tma_only(ep.kind) && ep.kind != kEpiSoftmaxGrad) || ep.kind == kEpiF32Add)
    return fail(MLP_EUNSUPPORTED, "batched GEMM: epilogue kind %d not supported", ep.kind);
  const int mode = g_pair_mode.load(std::memory_order_relaxed);
  const bool pair = mode == 1 || (mode < 0 && M > kBM);
  const uint32_t b_tile = pair ? GemmCfg<true>::kBLoadN : GemmCfg<false>::kBLoadN;
  CUtensorMap mA, mB, mC, mO0, mO1;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  int rc = a.mn_major ? make_map4(&mA, bf, 2, a.base, a.mn, a.k, a.ld, nb_h, a.h_stride, nb_s, a.s_stride, 64, kBK,
                                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B)
                      : make_map4(&mA, bf, 2, a.base, a.k, a.mn, a.ld, nb_h, a.h_stride, nb_s, a.s_stride, kBK, kBM,
                                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  if (rc) return rc;
  rc = b.mn_major ? make_map4(&mB, bf, 2, b.base, b.mn, b.k, b.ld, nb_h, b.h_stride, nb_s, b.s_stride, 64, kBK,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B)
                  : make_map4(&mB, bf, 2, b.base, b.k, b.mn, b.ld, nb_h, b.h_stride, nb_s, b.s_stride, kBK, b_tile,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  if (rc) return rc;
  memset(&mC, 0, sizeof(mC));
  memset(&mO0, 0, sizeof(mO0));
  memset(&mO1, 0, sizeof(mO1));
  if (epi_f32_out(ep.kind))
    rc = make_map4(&mC, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, out.base, out.cols, out.rows, out.ld, nb_h, out.h_stride,
                   nb_s, out.s_stride, 32, 32, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE);
  else
    rc = make_map4(&mO0, bf, 2, out.base, out.cols, out.rows, out.ld, nb_h, out.h_stride, nb_s, out.s_stride, 32, 32,
                   CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE);
  if (rc) return rc;
  if (ep.kind == kEpiSoftmaxGrad)  // P, laid out like the output, read by the epilogue through TMA
    rc = make_map4(&mO1, bf, 2, ep.in0, out.cols, out.rows, out.ld, nb_h, out.h_stride, nb_s, out.s_stride, 32, 32,
                   CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE);
  if (rc) return rc;
  const int raster_n_fast = M > N ? 1 : 0;
  const int batch = nb_h * nb_s;
  if (!a.mn_major && b.mn_major)
    return pair ? launch_gemm_t<false, true, true, true>(st, mA, mB, mC, mO0, mO1, M, N, K, ep, raster_n_fast, 0, 0,
                                                         stream, trace_kind, batch, nb_h, causal)
                : launch_gemm_t<false, true, false, true>(st, mA, mB, mC, mO0, mO1, M, N, K, ep, raster_n_fast, 0, 0,
                                                          stream, trace_kind, batch, nb_h, causal);
  if (!a.mn_major && !b.mn_major)
    return pair ? launch_gemm_t<false, false, true, true>(st, mA, mB, mC, mO0, mO1, M, N, K, ep, raster_n_fast, 0, 0,
                                                          stream, trace_kind, batch, nb_h, causal)
                : launch_gemm_t<false, false, false, true>(st, mA, mB, mC, mO0, mO1, M, N, K, ep, raster_n_fast, 0, 0,
                                                           stream, trace_kind, batch, nb_h, causal);
  if (a.mn_major && b.mn_major)
    return pair ? launch_gemm_t<true, true, true, true>(st, mA, mB, mC, mO0, mO1, M, N, K, ep, raster_n_fast, 0, 0,
                                                        stream, trace_kind, batch, nb_h, causal)
                : launch_gemm_t<true, true, false, true>(st, mA, mB, mC, mO0, mO1, M, N, K, ep, raster_n_fast, 0, 0,
                                                         stream, trace_kind, batch, nb_h, causal);
  return fail(MLP_EUNSUPPORTED, "batched GEMM: operand layout combination not instantiated");
}
