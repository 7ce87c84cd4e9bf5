// Persistent, warp-specialised tcgen05 GEMM for sm_103a with fused epilogues.
//
//   D[M, N] = sum_k A(m, k) * B(n, k)       (bf16 operands, fp32 accumulator in TMEM)
//
// Operands live row-major in HBM; each may be K-major (k contiguous) or MN-major
// (m or n contiguous), so the six contractions of the MLP block's forward and
// backward never materialise a transpose.  Each CTA owns 128 x 256 of D per
// tile, with BK = 64 (one 128-byte swizzle atom of bf16 along the contiguous
// dimension).  Two variants:
//   single CTA  tcgen05.mma.cta_group::1, M = 128, N = 256; 4-stage ring of 48 KB.
//   CTA pair    a cluster of two CTAs computes a 256 x 256 tile with
//               tcgen05.mma.cta_group::2 issued by the even CTA: each CTA loads
//               its own 128 rows of A and its half (128) of B's columns, so per
//               SM the B traffic (smem and L2) halves; 6-stage ring of 32 KB.
// (Batched GEMMs: 3 and 5 stages, see GemmCfg.)  The grid is persistent.  An
// item of work is a tile, or, in the split tail of a GEMM whose last wave would
// be at most half full, one half of a tile's reduction (see EpiParams).  CTAs
// (pairs) take items either round-robin (static) or, with a tile counter in
// global memory, each the next one when it is ready for it (dynamic: the CTAs
// that share an operand stripe then start it together instead of drifting apart
// over the waves of a long GEMM, so the stripe is read from DRAM once and served
// from L2 to the others).
//
// Warp roles (192 threads, or 320 in the wide configuration; one CTA per SM):
//   warp 0      TMA producer: loads A/B k-blocks into the smem ring.
//   warp 1      TMEM owner and (even CTA) MMA issuer: one thread issues
//               tcgen05.mma; the accumulator is double-buffered (2 x 256 fp32
//               columns of TMEM) so the epilogue of tile j overlaps the main
//               loop of tile j+1.
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (warp w reads TMEM lane
//               quarter w % 4, i.e. tile rows 32*(w%4) .. +31; the wide
//               configuration has warps 2..9, two per quarter, each on half the
//               columns), fused element-wise
//               work, TMA stores.  The 8 column blocks of a tile leave paced
//               against the producer's progress through the next tile: a burst
//               of output stores (fp32 gradients above all) starves that tile's
//               operand copies, and the tensor pipe with them.
// Every mbarrier wait is bounded; on timeout the kernel records kStatusTimeout in
// the status word, drains its own copies and MMAs, frees TMEM and returns.
#pragma once
#include <cstdint>
#include <cuda.h>

#include "block_math.cuh"
#include "ptx.cuh"

namespace gbmlp {

constexpr int kBM = 128;   // rows of D per CTA per tile
constexpr int kBN = 256;   // columns of D per tile (the MMA's N)
constexpr int kBK = 64;
constexpr uint32_t kABytes = kBM * kBK * 2;     // 16 KB
constexpr uint32_t kChunkBytes = 64 * kBK * 2;  // one 64 x BK box of an MN-major operand
constexpr uint32_t kTmemCols = 2 * kBN;         // double-buffered accumulator
// Dynamic tile scheduling: the even CTA's producer draws items from a counter in
// global memory and hands them to every other role of both CTAs through a ring of
// kItemDepth slots in shared memory.
constexpr int kItemDepth = 4;
// Outputs leave through TMA: each epilogue warp stages 32 rows x 32 columns in
// one of two buffers and issues a bulk store (or, for fp32, a bulk reduce-add).
// fp32 boxes are 4 KB with a 128-byte swizzle.
// bf16 outputs likewise, as 32 x 32 boxes with a 64-byte swizzle (two outputs
// per buffer for the GeLU epilogue, which writes U and Y).
constexpr uint32_t kOutBoxBytes = 32 * 32 * 4;
constexpr uint32_t kOutBoxBf16Bytes = 32 * 32 * 2;
// Longest an epilogue warp waits for the main loop before it stores anyway.
constexpr uint64_t kPaceLimitNs = 200000;

// Staged epilogue inputs (see the epilogue) live in the free halves of the two
// output buffers of each epilogue warp: a ring of kInDepth = 2 boxes.
// WIDE configurations (the batched attention products, whose reductions run over
// a head size, and plain GEMMs with reductions under 16 k-blocks: their time is in
// the epilogue) run 8 epilogue warps, two per TMEM lane quarter, each on half of
// the tile's columns, and pay for the extra staging with a shorter ring.
template <bool PAIR, bool WIDE = false>
struct GemmCfg {
  static constexpr int kEpiWarps = WIDE ? 8 : 4;
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  static constexpr int kStages = WIDE ? (PAIR ? 5 : 3) : (PAIR ? 6 : 4);
  static constexpr int kBLoadN = PAIR ? kBN / 2 : kBN;      // B rows (N) this CTA loads per stage
  static constexpr int kTileM = PAIR ? 2 * kBM : kBM;       // rows of D per tile
  static constexpr uint32_t kBBytes = kBLoadN * kBK * 2;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr int kInDepth = 2;
  static constexpr uint32_t kOutBytes = kEpiWarps * 2 * kOutBoxBytes;  // 2 staging buffers per epilogue warp
  static constexpr size_t kSmemBytes = (size_t)kStages * kStageBytes + kOutBytes + 1024 /*align*/ + 512 /*barriers*/;
};
static_assert(GemmCfg<true>::kSmemBytes <= 232448 && GemmCfg<false>::kSmemBytes <= 232448 &&
                  GemmCfg<true, true>::kSmemBytes <= 232448 && GemmCfg<false, true>::kSmemBytes <= 232448,
              "smem budget");

enum CausalMode : int { kCausalNone = 0, kCausalSkipUpper = 1, kCausalKUpTo = 2, kCausalKFrom = 3 };

enum EpiKind : int {
  kEpiGelu = 0,      // U = acc + bias (bf16), Y = GeLU(acc + bias) (bf16)
  kEpiF32Store = 1,  // G = acc (fp32)
  kEpiF32Add = 2,    // G += acc (fp32 read-modify-write)
  kEpiDropRes = 3,   // O = R + dropout((G ? G : 0) + acc + bias) (bf16)
  kEpiDGelu = 4,     // dU = acc * GeLU'(U) (bf16)
  kEpiResAdd = 5,    // dX = (G ? G : 0) + acc + (R ? R : 0) (bf16)
  kEpiBias = 6,      // out = acc + bias (bf16)
  kEpiStore = 7,     // out = acc (bf16)
  kEpiScaleMask = 8,    // G = (column > row ? -inf : alpha * acc) (fp32; causal attention scores)
  kEpiSoftmaxGrad = 9   // dS = P * (acc - delta[batch][row]) * alpha (bf16; batched; P staged by TMA)
};

// Epilogues whose output is fp32 (written through the fp32 TMA map tmC).
__host__ __device__ constexpr bool epi_f32_out(int kind) {
  return kind == kEpiF32Store || kind == kEpiF32Add || kind == kEpiScaleMask;
}
// Epilogues that read no tensor through plain pointers (usable in batched GEMMs).
__host__ __device__ constexpr bool epi_tma_only(int kind) {
  return epi_f32_out(kind) || kind == kEpiStore;
}
// Epilogues that read a bf16 input (in0) through a TMA-staged box (map tmO1).
__host__ __device__ constexpr bool epi_staged_input(int kind) {
  return kind == kEpiDGelu || kind == kEpiDropRes || kind == kEpiResAdd || kind == kEpiSoftmaxGrad;
}

struct EpiParams {
  int kind;
  int64_t ld;                 // leading dimension (elements) shared by every tensor the epilogue touches
  float* g_out;               // fp32 output (F32Store / F32Add)
  const float* g_in;          // fp32 partial sum read by DropRes / ResAdd (may be null); SoftmaxGrad: delta,
                              // ld floats per batch matrix
  uint16_t* out0;             // bf16 output: U / O / dU / dX
  uint16_t* out1;             // bf16 output: Y
  const uint16_t* in0;        // bf16 input: R (DropRes, ResAdd) or U (DGelu); may be null for ResAdd
  const uint16_t* bias;       // bias vector indexed by output column
  float alpha;                // scale of kEpiScaleMask and kEpiSoftmaxGrad
  DropoutParams drop;
  int pace;                   // 1: pace the output stores against the next tile's main loop
  // Split tail (bf16 epilogues of plain GEMMs): tiles [split_base, num_tiles) are
  // computed as two halves of the reduction by two CTAs (pairs); each half writes
  // its fp32 partial to split_ws and counts itself in split_flags, and the second
  // to arrive adds the other's partial to its own and runs the epilogue.
  int split_base;
  float* split_ws;            // kSplitSlots x 2 halves x (32 x 256) fp32
  int* split_flags;           // kSplitSlots counters, 0 between launches
};
// Slots of the split tail: (tile, CTA of the pair, epilogue warp) triples.
constexpr int kSplitSlots = 304;
constexpr int kSplitSlotFloats = 32 * 256;

__device__ __forceinline__ void ld_bf16x8(const uint16_t* p, float (&v)[8]) {
  const uint4 q = *reinterpret_cast<const uint4*>(p);
  v[0] = bf16lo(q.x); v[1] = bf16hi(q.x);
  v[2] = bf16lo(q.y); v[3] = bf16hi(q.y);
  v[4] = bf16lo(q.z); v[5] = bf16hi(q.z);
  v[6] = bf16lo(q.w); v[7] = bf16hi(q.w);
}

__device__ __forceinline__ void ld_f32x8(const float* p, float (&v)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0];
  const float4 b = reinterpret_cast<const float4*>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// The bf16 input in0 of lane `lane`'s row, columns [8 g, 8 g + 8) of a 32 x 32
// box staged by TMA with the 64-byte swizzle.
__device__ __forceinline__ void ld_staged_bf16x8(const uint8_t* box, int lane, int g, float (&v)[8]) {
  const uint4 q = *reinterpret_cast<const uint4*>(box + lane * 64 + ((g ^ ((lane >> 1) & 3)) << 4));
  v[0] = bf16lo(q.x); v[1] = bf16hi(q.x);
  v[2] = bf16lo(q.y); v[3] = bf16hi(q.y);
  v[4] = bf16lo(q.z); v[5] = bf16hi(q.z);
  v[6] = bf16lo(q.w); v[7] = bf16hi(q.w);
}

// One thread, one row, 32 accumulator columns [col0, col0 + 32); N % 8 == 0.
// Computes the bf16 output(s) of the fused epilogue, packed two per word:
// o0 = U / O / dU / dX, o1 = Y (GeLU only).  Inputs are read only inside the
// tensor (row < M, col < N); out-of-range lanes produce values the TMA store clips.
// in_box: in0's 32 x 32 box for this warp and column block, staged in shared
// memory by TMA (zero outside the tensor), or null to read in0 from global memory.
template <int KIND>
__device__ __forceinline__ void epilogue_values(const EpiParams& ep, int64_t row, int col0, const uint32_t (&r)[32],
                                                int M, int N, uint32_t (&o0)[16], uint32_t (&o1)[16],
                                                const uint8_t* in_box) {
  const bool row_ok = row < M;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const int col = col0 + 8 * g;
    const bool col_ok = col < N;
    const bool ok = row_ok && col_ok;
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = __uint_as_float(r[8 * g + j]);
    const int64_t off = row * ep.ld + col;
    if constexpr (KIND == kEpiGelu) {
      float bb[8] = {0, 0, 0, 0, 0, 0, 0, 0}, y[8];
      if (col_ok) ld_bf16x8(ep.bias + col, bb);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        v[j] += bb[j];
        y[j] = gelu_f(v[j]);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        o0[4 * g + j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
        o1[4 * g + j] = pack_bf16x2(y[2 * j], y[2 * j + 1]);
      }
    } else if constexpr (KIND == kEpiDropRes) {
      float bb[8] = {0, 0, 0, 0, 0, 0, 0, 0}, res[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (ok && ep.g_in != nullptr) {
        float z[8];
        ld_f32x8(ep.g_in + off, z);
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = z[j] + v[j];
      }
      if (col_ok) ld_bf16x8(ep.bias + col, bb);
      if (in_box != nullptr)
        ld_staged_bf16x8(in_box, lane, g, res);
      else if (ok)
        ld_bf16x8(ep.in0 + off, res);
      const uint32_t keep = dropout_keep8(ep.drop, row, col);
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = res[j] + (((keep >> j) & 1u) ? (v[j] + bb[j]) * ep.drop.scale : 0.0f);
#pragma unroll
      for (int j = 0; j < 4; ++j) o0[4 * g + j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
    } else if constexpr (KIND == kEpiDGelu) {
      float u[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (in_box != nullptr)
        ld_staged_bf16x8(in_box, lane, g, u);
      else if (ok)
        ld_bf16x8(ep.in0 + off, u);
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] *= gelu_prime_f(u[j]);
#pragma unroll
      for (int j = 0; j < 4; ++j) o0[4 * g + j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
    } else if constexpr (KIND == kEpiBias) {
      float bb[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (col_ok) ld_bf16x8(ep.bias + col, bb);
#pragma unroll
      for (int j = 0; j < 4; ++j) o0[4 * g + j] = pack_bf16x2(v[2 * j] + bb[2 * j], v[2 * j + 1] + bb[2 * j + 1]);
    } else if constexpr (KIND == kEpiStore) {
#pragma unroll
      for (int j = 0; j < 4; ++j) o0[4 * g + j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
    } else {  // kEpiResAdd
      if (ok && ep.g_in != nullptr) {
        float z[8];
        ld_f32x8(ep.g_in + off, z);
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = z[j] + v[j];
      }
      if (ep.in0 != nullptr && (ok || in_box != nullptr)) {
        float res[8];
        if (in_box != nullptr)
          ld_staged_bf16x8(in_box, lane, g, res);
        else
          ld_bf16x8(ep.in0 + off, res);
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] += res[j];
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) o0[4 * g + j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
    }
  }
}

__device__ __forceinline__ void epilogue_dispatch(const EpiParams& ep, int64_t row, int col0, const uint32_t (&r)[32],
                                                  int M, int N, uint32_t (&o0)[16], uint32_t (&o1)[16],
                                                  const uint8_t* in_box) {
  switch (ep.kind) {
    case kEpiGelu: epilogue_values<kEpiGelu>(ep, row, col0, r, M, N, o0, o1, in_box); break;
    case kEpiDropRes: epilogue_values<kEpiDropRes>(ep, row, col0, r, M, N, o0, o1, in_box); break;
    case kEpiDGelu: epilogue_values<kEpiDGelu>(ep, row, col0, r, M, N, o0, o1, in_box); break;
    case kEpiBias: epilogue_values<kEpiBias>(ep, row, col0, r, M, N, o0, o1, in_box); break;
    case kEpiStore: epilogue_values<kEpiStore>(ep, row, col0, r, M, N, o0, o1, in_box); break;
    default: epilogue_values<kEpiResAdd>(ep, row, col0, r, M, N, o0, o1, in_box); break;
  }
}

__device__ __forceinline__ void record_status(int* status, int code, int site) {
  if (status != nullptr) {
    if (atomicCAS(status, 0, code) == 0) status[1] = site;
  }
}

// A_MN / B_MN: operand stored MN-major (true) or K-major (false).
// PAIR: launched as clusters of two CTAs (see the file comment).
// tmC: fp32 output map (box 32 x 32, 128-byte swizzle) used by kEpiF32Store / kEpiF32Add.
// tmO0 / tmO1: bf16 output maps (box 32 x 32, 64-byte swizzle) of out0 / out1.
// raster_n_fast: tiles are visited with N varying fastest (else M fastest), so that
// the operand re-read across the sweep is the smaller one and stays in L2.
// group: if > 0, the fast dimension is swept in groups of `group` blocks: all
// tiles of those blocks (across the whole slow dimension) come before the next
// group, so that only `group` stripes of the smaller operand need to stay in L2
// while the larger operand streams past them.
// l2_hints: L2 policy of the A loads (bits 0-1), the B loads (bits 2-3) and the
// output stores (bits 4-5), an L2Hint each (kL2None: no hint).
// sched: null for the static round-robin order, else two ints in global memory,
// both 0 at launch: [0] the next item to hand out, [1] the CTAs (pairs) that have
// finished drawing; the last to finish sets both back to 0 for the next launch
// (which may not touch them before this grid completes: no late wait).
// BATCHED: `batch` independent GEMMs of the same M, N, K; every tensor map is 4-D
// (x, y, hb, sb) with batch b = sb * nb_h + hb; only TMA-only epilogues and the softmax gradient.
// causal (batched attention products, M and N or K indexing positions in one
// sequence): kCausalNone; kCausalSkipUpper skips tiles whose columns all lie
// after the tile's last row (the result there is never read); kCausalKUpTo stops
// each tile's reduction after its last row (A(m, k) = 0 for k > m);
// kCausalKFrom starts it at the tile's first row (A(m, k) = 0 for k < m).
template <bool A_MN, bool B_MN, bool PAIR, bool BATCHED, bool WIDE = false>
__global__ void __launch_bounds__(GemmCfg<PAIR, BATCHED || WIDE>::kThreads, 1)
    k_gemm_bf16_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmO0,
                   const __grid_constant__ CUtensorMap tmO1, int M, int N, int K, EpiParams ep, int raster_n_fast,
                   int group, int l2_hints, int batch, int nb_h, int causal, int late_wait, int* sched,
                   int* status) {
  using Cfg = GemmCfg<PAIR, BATCHED || WIDE>;
  constexpr int kStages = Cfg::kStages;
  constexpr int kEpiWarps = Cfg::kEpiWarps;
  constexpr int kInDepth = Cfg::kInDepth;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kABytes;
  uint8_t* sOut = sB + kStages * Cfg::kBBytes;  // 1024-aligned
  uint64_t* full = reinterpret_cast<uint64_t*>(sOut + Cfg::kOutBytes);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* mma_done = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  uint64_t* in_full = mma_done + 2;  // per epilogue warp, kInDepth: staged input boxes
  uint64_t* item_full = in_full + kEpiWarps * kInDepth;  // dynamic scheduling: item ring
  uint64_t* item_empty = item_full + kItemDepth;
  int* s_item = reinterpret_cast<int*>(item_empty + kItemDepth);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;     // 0 = the CTA that issues the MMAs
  const int unit = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;   // CTA pair or single CTA
  const int num_units = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  const int num_m = (M + Cfg::kTileM - 1) / Cfg::kTileM;
  const int num_n = (N + kBN - 1) / kBN;
  const int tiles_per_batch = num_m * num_n;
  const int num_tiles = tiles_per_batch * (BATCHED ? batch : 1);
  const int num_kb = (K + kBK - 1) / kBK;

  // A pipeline that broke in an earlier launch leaves the status word set; later
  // launches then skip their work so that a failure ends quickly.
  __shared__ int s_skip;
  // k-blocks whose copies this CTA's producer has issued, over all its tiles so far
  __shared__ uint32_t s_kb_issued;
  volatile uint32_t* kb_issued = &s_kb_issued;
  if (threadIdx.x == 0) {
    s_kb_issued = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], (PAIR ? 2 : 1) * kEpiWarps);  // one arrival per epilogue warp (of both CTAs)
    }
    mbar_init(mma_done, 1);
    for (int i = 0; i < kEpiWarps * kInDepth; ++i) mbar_init(&in_full[i], 1);
    for (int i = 0; i < kItemDepth; ++i) {
      mbar_init(&item_full[i], 1);
      // consumers: the MMA issuer and the epilogue warps of the even CTA; the
      // producer and the epilogue warps of the odd CTA (they arrive remotely)
      mbar_init(&item_empty[i], PAIR ? 2 + 2 * kEpiWarps : 1 + kEpiWarps);
    }
    fence_mbar_init();
  }
  const bool tma_out = epi_f32_out(ep.kind);
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (tma_out) {
      tma_prefetch_desc(&tmC);
    } else {
      tma_prefetch_desc(&tmO0);
      if (ep.kind == kEpiGelu || (ep.in0 != nullptr && epi_staged_input(ep.kind))) tma_prefetch_desc(&tmO1);
    }
  }
  if (warp == 1) {
    tmem_alloc<PAIR>(tmem_slot, kTmemCols);
    tmem_relinquish<PAIR>();
  }
  // Everything above touches only this CTA's own resources; from here on the
  // kernel reads what the previous kernel on the stream wrote.  With late_wait the
  // host guarantees that this launch reads nothing the immediately preceding
  // kernel writes and that kernel waited for its own predecessor before letting
  // this one start, so the main loop may overlap that kernel's tail; the wait
  // then comes before exit, so that this grid completes only after it.
  if (!late_wait) grid_dependency_wait();
  grid_launch_dependents();
  if (threadIdx.x == 0) s_skip = (status != nullptr && *reinterpret_cast<volatile int*>(status) != 0) ? 1 : 0;
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) {
    // both CTAs' barriers are initialised before either CTA signals the other's;
    // the skip decision is shared so both CTAs walk the same tiles
    cluster_sync();
  }
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  int skip = s_skip;
  if constexpr (PAIR) {
    int* peer_skip = static_cast<int*>(__cluster_map_shared_rank(static_cast<void*>(&s_skip), rank ^ 1u));
    skip |= *reinterpret_cast<volatile int*>(peer_skip);
    cluster_sync();  // the peer has read s_skip before anything else touches it
  }
  // Work items: tiles [0, split_base) whole, then each tile of the split tail as two
  // items, one per half of its reduction (see EpiParams).
  const int split_base =
      (!BATCHED && kEpiWarps == 4 && ep.split_ws != nullptr) ? min(ep.split_base, num_tiles) : num_tiles;
  const int num_items = split_base + 2 * (num_tiles - split_base);
  const int item_end = skip ? 0 : num_items;

  auto tile_origin = [&](int tile, int& m0, int& n0, int& hb, int& sb) {
    hb = 0;
    sb = 0;
    if constexpr (BATCHED) {
      const int b = tile / tiles_per_batch;
      tile -= b * tiles_per_batch;
      hb = b % nb_h;
      sb = b / nb_h;
    }
    // fast: blocks along the fast dimension; slow: along the other one
    const int n_fast = raster_n_fast ? num_n : num_m;
    const int n_slow = raster_n_fast ? num_m : num_n;
    const int g = group > 0 ? group : n_fast;
    const int gi = tile / (g * n_slow);             // group index
    const int gw = min(g, n_fast - gi * g);         // width of this group
    const int r = tile - gi * g * n_slow;
    const int fast = gi * g + r % gw;
    const int slow = r / gw;
    const int mb = raster_n_fast ? slow : fast;
    const int nb = raster_n_fast ? fast : slow;
    m0 = mb * Cfg::kTileM + (int)rank * kBM;  // this CTA's first row
    n0 = nb * kBN;
  };
  // causal structure of the batched attention products (see above); decided per
  // tile from the tile's row range, identically in every role and in both CTAs
  auto tile_rows = [&](int m0) { return m0 - (int)rank * kBM; };  // first row of the whole tile
  auto skip_tile = [&](int m0, int n0) {
    return causal == kCausalSkipUpper && n0 >= tile_rows(m0) + Cfg::kTileM;
  };
  auto kb_range = [&](int m0, int& kb0, int& kb1) {
    kb0 = 0;
    kb1 = num_kb;
    if (causal == kCausalKUpTo) {
      const int k_end = min(K, tile_rows(m0) + Cfg::kTileM);
      kb1 = (k_end + kBK - 1) / kBK;
    } else if (causal == kCausalKFrom) {
      kb0 = tile_rows(m0) / kBK;
    }
  };

  // Decodes a work item into its tile's origin, its k-block range and its half
  // of the reduction (-1: the whole tile); false if the tile is skipped.
  auto item_info = [&](int item, int& m0, int& n0, int& hb, int& sb, int& kb0, int& kb1, int& half) -> bool {
    int tile = item;
    half = -1;
    if (item >= split_base) {
      tile = split_base + ((item - split_base) >> 1);
      half = (item - split_base) & 1;
    }
    tile_origin(tile, m0, n0, hb, sb);
    if (skip_tile(m0, n0)) return false;
    kb_range(m0, kb0, kb1);
    if (half >= 0) {
      const int mid = (kb0 + kb1) / 2;
      if (half == 0)
        kb1 = mid;
      else
        kb0 = mid;
    }
    return true;
  };

  // ---- the sequence of items each role works through.  Item n of this CTA
  // (pair): static, unit + n * num_units; dynamic, the n-th item the even CTA's
  // producer drew from the counter, read from ring slot n % kItemDepth.  -1 ends
  // the sequence.  Every wait is bounded; a role that gives up records the
  // timeout and sees -1.
  const bool dynamic = sched != nullptr;
  // Even CTA's producer: draw item n from the counter and publish it to both CTAs.
  auto draw_item = [&](uint32_t n) -> int {
    const int slot = (int)(n % kItemDepth);
    if (!mbar_wait_cluster(&item_empty[slot], ((n / kItemDepth) & 1) ^ 1)) {
      record_status(status, kStatusTimeout, 8);
      return -1;
    }
    int item = atomicAdd(&sched[0], 1);
    if (item >= item_end) item = -1;
    s_item[slot] = item;
    if constexpr (PAIR) {
      asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(mapa_shared(smem_u32(&s_item[slot]), 1)), "r"(item)
                   : "memory");
      mbar_arrive_cluster(mapa_shared(smem_u32(&item_full[slot]), 1));
    }
    mbar_arrive(&item_full[slot]);
    return item;
  };
  // Every other role: item n as published.  release: free the slot (one arrival
  // per role: `whole_warp` roles call this from all 32 lanes and lane 0 arrives
  // once they have all read it; single-thread roles arrive themselves); a peek
  // (release = false) leaves the slot to the later read that releases it.
  auto read_item = [&](uint32_t n, bool release, bool whole_warp) -> int {
    const int slot = (int)(n % kItemDepth);
    if (!mbar_wait_cluster(&item_full[slot], (n / kItemDepth) & 1)) {
      record_status(status, kStatusTimeout, 9);
      return -1;
    }
    const int item = *reinterpret_cast<volatile int*>(&s_item[slot]);
    if (release) {
      if (whole_warp) __syncwarp();
      if (!whole_warp || (threadIdx.x & 31) == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&item_empty[slot]), 0));
    }
    return item;
  };
  auto static_item = [&](uint32_t n) -> int {
    const int item = unit + (int)n * num_units;
    return item < item_end ? item : -1;
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      const int ha = l2_hints & 3, hb = (l2_hints >> 2) & 3;
      const uint64_t pol_a = l2_policy(ha);
      const uint64_t pol_b = l2_policy(hb);
      uint32_t issued[kStages];
#pragma unroll
      for (int s = 0; s < kStages; ++s) issued[s] = 0;
      uint32_t n_issued = 0;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (uint32_t n_item = 0; ok; ++n_item) {
        const int item = !dynamic ? static_item(n_item) : rank == 0 ? draw_item(n_item) : read_item(n_item, true, false);
        if (item < 0) break;
        int m0, n0, hb, sb, kb0, kb1, half;
        if (!item_info(item, m0, n0, hb, sb, kb0, kb1, half)) continue;
        const int b_n0 = n0 + (PAIR ? (int)rank * Cfg::kBLoadN : 0);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1)) {
            record_status(status, kStatusTimeout, 1);
            ok = false;
            break;
          }
          const int k0 = kb * kBK;
          uint8_t* a_dst = sA + stage * kABytes;
          uint8_t* b_dst = sB + stage * Cfg::kBBytes;
          if constexpr (BATCHED) {
            if constexpr (PAIR) {
              const uint32_t bar = mapa_shared(smem_u32(&full[stage]), 0);
              if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * Cfg::kStageBytes);
              if constexpr (A_MN) {
#pragma unroll
                for (int j = 0; j < kBM / 64; ++j)
                  tma_load_4d_pair(a_dst + j * kChunkBytes, &tmA, bar, m0 + 64 * j, k0, hb, sb);
              } else {
                tma_load_4d_pair(a_dst, &tmA, bar, k0, m0, hb, sb);
              }
              if constexpr (B_MN) {
#pragma unroll
                for (int j = 0; j < Cfg::kBLoadN / 64; ++j)
                  tma_load_4d_pair(b_dst + j * kChunkBytes, &tmB, bar, b_n0 + 64 * j, k0, hb, sb);
              } else {
                tma_load_4d_pair(b_dst, &tmB, bar, k0, b_n0, hb, sb);
              }
            } else {
              mbar_arrive_expect_tx(&full[stage], Cfg::kStageBytes);
              if constexpr (A_MN) {
#pragma unroll
                for (int j = 0; j < kBM / 64; ++j)
                  tma_load_4d(a_dst + j * kChunkBytes, &tmA, &full[stage], m0 + 64 * j, k0, hb, sb);
              } else {
                tma_load_4d(a_dst, &tmA, &full[stage], k0, m0, hb, sb);
              }
              if constexpr (B_MN) {
#pragma unroll
                for (int j = 0; j < Cfg::kBLoadN / 64; ++j)
                  tma_load_4d(b_dst + j * kChunkBytes, &tmB, &full[stage], b_n0 + 64 * j, k0, hb, sb);
              } else {
                tma_load_4d(b_dst, &tmB, &full[stage], k0, b_n0, hb, sb);
              }
            }
          } else if constexpr (PAIR) {
            // both CTAs' copies complete on the even CTA's barrier, which expects both
            const uint32_t bar = mapa_shared(smem_u32(&full[stage]), 0);
            if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * Cfg::kStageBytes);
            if constexpr (A_MN) {
#pragma unroll
              for (int j = 0; j < kBM / 64; ++j) tma_load_2d_pair(a_dst + j * kChunkBytes, &tmA, bar, m0 + 64 * j, k0, pol_a, ha != kL2None);
            } else {
              tma_load_2d_pair(a_dst, &tmA, bar, k0, m0, pol_a, ha != kL2None);
            }
            if constexpr (B_MN) {
#pragma unroll
              for (int j = 0; j < Cfg::kBLoadN / 64; ++j)
                tma_load_2d_pair(b_dst + j * kChunkBytes, &tmB, bar, b_n0 + 64 * j, k0, pol_b, hb != kL2None);
            } else {
              tma_load_2d_pair(b_dst, &tmB, bar, k0, b_n0, pol_b, hb != kL2None);
            }
          } else {
            mbar_arrive_expect_tx(&full[stage], Cfg::kStageBytes);
            if constexpr (A_MN) {
#pragma unroll
              for (int j = 0; j < kBM / 64; ++j)
                tma_load_2d(a_dst + j * kChunkBytes, &tmA, &full[stage], m0 + 64 * j, k0, pol_a, ha != kL2None);
            } else {
              tma_load_2d(a_dst, &tmA, &full[stage], k0, m0, pol_a, ha != kL2None);
            }
            if constexpr (B_MN) {
#pragma unroll
              for (int j = 0; j < Cfg::kBLoadN / 64; ++j)
                tma_load_2d(b_dst + j * kChunkBytes, &tmB, &full[stage], b_n0 + 64 * j, k0, pol_b, hb != kL2None);
            } else {
              tma_load_2d(b_dst, &tmB, &full[stage], k0, b_n0, pol_b, hb != kL2None);
            }
          }
          ++issued[stage];
          *kb_issued = ++n_issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // Drain: every copy this CTA issued has landed before the CTA may exit.
      if (!PAIR || rank == 0) {
        for (int s = 0; s < kStages; ++s) {
          if (issued[s] > 0 && !(PAIR ? mbar_wait_cluster(&full[s], (issued[s] - 1) & 1)
                                      : mbar_wait(&full[s], (issued[s] - 1) & 1)))
            record_status(status, kStatusTimeout, 2);
        }
      } else if (!ok) {
        // the odd CTA's copies complete on the even CTA's barrier; after a failure
        // give any copy still in flight time to land (bounded)
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 2000000ull) __nanosleep(10000);
      }
      if (dynamic && rank == 0) {
        // this CTA (pair) draws no more; the last one to finish resets the counter
        __threadfence();
        if (atomicAdd(&sched[1], 1) == num_units - 1) {
          atomicExch(&sched[0], 0);
          atomicExch(&sched[1], 0);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = make_idesc_bf16(PAIR ? 2 * kBM : kBM, kBN, A_MN, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (uint32_t n_item = 0; ok; ++n_item) {
        const int item = dynamic ? read_item(n_item, true, false) : static_item(n_item);
        if (item < 0) break;
        int m0, n0, hb, sb, kb0, kb1, half;
        if (!item_info(item, m0, n0, hb, sb, kb0, kb1, half)) continue;
        if (!(PAIR ? mbar_wait_cluster(&acc_empty[acc], acc_phase ^ 1) : mbar_wait(&acc_empty[acc], acc_phase ^ 1))) {
          record_status(status, kStatusTimeout, 3);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * kBN;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!(PAIR ? mbar_wait_cluster(&full[stage], phase) : mbar_wait(&full[stage], phase))) {
            record_status(status, kStatusTimeout, 4);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + stage * kABytes);
          const uint32_t b_base = smem_u32(sB + stage * Cfg::kBBytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t adesc = A_MN ? make_sdesc_sw128(a_base + kk * 2048, kChunkBytes, 1024)
                                        : make_sdesc_sw128(a_base + kk * 32, 16, 1024);
            const uint64_t bdesc = B_MN ? make_sdesc_sw128(b_base + kk * 2048, kChunkBytes, 1024)
                                        : make_sdesc_sw128(b_base + kk * 32, 16, 1024);
            const uint32_t accumulate = (kb != kb0 || kk != 0) ? 1u : 0u;
            if constexpr (PAIR)
              umma_bf16_pair(d_tmem, adesc, bdesc, idesc, accumulate);
            else
              umma_bf16(d_tmem, adesc, bdesc, idesc, accumulate);
          }
          // the smem stage (of both CTAs) is free once these MMAs have read it
          if constexpr (PAIR)
            umma_commit_pair(&empty[stage], 0x3);
          else
            umma_commit(&empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        // accumulator ready for the epilogue warps (of both CTAs)
        if constexpr (PAIR)
          umma_commit_pair(&acc_full[acc], 0x3);
        else
          umma_commit(&acc_full[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      if constexpr (PAIR)
        umma_commit_pair(mma_done, 0x1);
      else
        umma_commit(mma_done);
      if (!mbar_wait(mma_done, 0)) record_status(status, kStatusTimeout, 5);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int quarter = warp & 3;
    const int row_in_tile = quarter * 32 + lane;
    // this warp's columns of each tile: all 256, or one half (8 epilogue warps)
    const int col_begin = kEpiWarps == 8 ? ((warp - 2) >> 2) * (kBN / 2) : 0;
    const int col_end = col_begin + kBN * 4 / kEpiWarps;
    uint8_t* my_out = sOut + (warp - 2) * 2 * kOutBoxBytes;
    uint32_t n_out = 0;  // boxes this warp has issued
    const int hout = (l2_hints >> 4) & 3;
    const uint64_t pol_out = l2_policy(hout);
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t kb_end = 0;  // the producer's k-block count once this tile's copies are all issued
    // Epilogues with a bf16 input in0 (U for GeLU', R for dropout + residual, dO
    // for the input gradient, P for the softmax gradient of the attention
    // products): the warp's 32 x 32 boxes of it are fetched by TMA (map tmO1)
    // through a ring of kInDepth buffers (the free halves of its output buffers),
    // kInDepth column blocks ahead, so the epilogue never waits on scattered global
    // loads.  A buffer is refilled only after the warp has read it and written its
    // output box.
    const bool prefetch_in = ep.in0 != nullptr && epi_staged_input(ep.kind) && (!BATCHED || ep.kind == kEpiSoftmaxGrad);
    uint64_t* my_in_full = in_full + kInDepth * (warp - 2);
    uint32_t n_in = 0;  // input boxes this warp has requested
    auto in_box = [&](uint32_t i) { return my_out + (i % kInDepth) * kOutBoxBytes + kOutBoxBf16Bytes; };
    auto request_in = [&](int x, int y, int hb, int sb) {
      if (lane == 0) {
        uint64_t* bar = &my_in_full[n_in % kInDepth];
        mbar_arrive_expect_tx(bar, kOutBoxBf16Bytes);
        if constexpr (BATCHED)
          tma_load_4d(in_box(n_in), &tmO1, bar, x, y, hb, sb);
        else
          tma_load_2d(in_box(n_in), &tmO1, bar, x, y, 0, false);
      }
      ++n_in;
    };
    auto wait_in = [&](uint32_t i) {
      if (!mbar_wait(&my_in_full[i % kInDepth], (i / kInDepth) & 1)) record_status(status, kStatusTimeout, 7);
    };
    for (uint32_t n_item = 0;; ++n_item) {
      const int item = dynamic ? read_item(n_item, true, true) : static_item(n_item);
      if (item < 0) break;
      int m0, n0, hb, sb, kb0, kb1, half;
      if (!item_info(item, m0, n0, hb, sb, kb0, kb1, half)) continue;
      kb_end += (uint32_t)max(kb1 - kb0, 0);
      // Reduction length of this CTA's next item, whose main loop these stores
      // are spread over (0: no next item, the stores go out at once).  With the
      // dynamic order the next item is drawn while this one's copies are issued,
      // long before this epilogue, so the peek does not wait in practice.
      uint32_t nkb_next = 0;
      const int next = dynamic ? read_item(n_item + 1, false, true) : static_item(n_item + 1);
      if (next >= 0) {
        int m1, n1, hb1, sb1, a0, a1, half1;
        if (item_info(next, m1, n1, hb1, sb1, a0, a1, half1)) nkb_next = (uint32_t)max(a1 - a0, 0);
      }
      // column blocks of this warp that produce output (the rest are clipped)
      const bool rows_in = m0 + quarter * 32 < M;
      const int n_blocks = (prefetch_in && rows_in && n0 + col_begin < N)
                               ? min((col_end - col_begin) / 32, (N - n0 - col_begin + 31) / 32) : 0;
      uint32_t n_in_used = n_in;  // index of the next input box to consume
      const int n_first = min(n_blocks, kInDepth);
      for (int q = 0; q < n_first; ++q) request_in(n0 + col_begin + 32 * q, m0 + quarter * 32, hb, sb);
      if (!(PAIR ? mbar_wait_cluster(&acc_full[acc], acc_phase) : mbar_wait(&acc_full[acc], acc_phase))) {
        record_status(status, kStatusTimeout, 6);
        break;
      }
      tc_fence_after();
      const int64_t row = (int64_t)m0 + row_in_tile;
      const uint32_t t_row = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * kBN);
      // Split tail: publish this half's partial (this warp's 32 rows x 256 columns),
      // count this half in; the half that arrives second adds the other's partial
      // to its own below and writes the output, the first is done.  fp32 addition
      // commutes, so the result does not depend on which half arrives second.
      const float* other = nullptr;
      bool finisher = true;
      if (half >= 0) {
        const int slot = (((item - split_base) >> 1) * (PAIR ? 2 : 1) + (int)rank) * 4 + quarter;
        float* mine = ep.split_ws + (size_t)(2 * slot + half) * kSplitSlotFloats + lane * 256;
#pragma unroll 1
        for (int c0 = 0; c0 < kBN; c0 += 32) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(t_row + c0, r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<uint4*>(mine + c0 + 4 * j) = make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
        }
        __threadfence();
        __syncwarp();
        int before = 0;
        if (lane == 0) before = atomicAdd(&ep.split_flags[slot], 1);
        before = __shfl_sync(0xffffffffu, before, 0);
        finisher = before == 1;
        if (finisher) {
          __threadfence();
          if (lane == 0) ep.split_flags[slot] = 0;  // ready for the next launch
          other = ep.split_ws + (size_t)(2 * slot + (half ^ 1)) * kSplitSlotFloats + lane * 256;
        } else {
          // no output from this half: retire the input boxes requested for it
          for (int q = 0; q < n_first; ++q) wait_in(n_in_used++);
        }
      }
      // One column block (32 columns) of this warp's rows: r holds its accumulator.
      auto pace_block = [&](int c0) {
        if (ep.pace && nkb_next > 0 && c0 > 0) {
          // Pace the output: column block c0 / 32 (of 8) leaves once the producer is
          // about (3 / 32) * (c0 / 32) of the way through the next tile's copies, so
          // the stores spread over two thirds of that main loop instead of competing
          // with its operand copies in one burst.  The target is always reached (the
          // next tile's copies do not depend on this epilogue); the wait is bounded
          // all the same and only delays.
          const uint32_t lead = min(nkb_next, (uint32_t)kStages + ((uint32_t)(c0 >> 5) * nkb_next * 3u) / 32u);
          if (lane == 0) {
            const uint64_t t0 = globaltimer_ns();
            while (*kb_issued < kb_end + lead && globaltimer_ns() - t0 < kPaceLimitNs) __nanosleep(128);
          }
          __syncwarp();
        }
      };
      auto out_block = [&](int c0, uint32_t (&r)[32]) {
        if (other != nullptr) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 o = __ldcg(reinterpret_cast<const float4*>(other + c0 + 4 * j));
            r[4 * j] = __float_as_uint(__uint_as_float(r[4 * j]) + o.x);
            r[4 * j + 1] = __float_as_uint(__uint_as_float(r[4 * j + 1]) + o.y);
            r[4 * j + 2] = __float_as_uint(__uint_as_float(r[4 * j + 2]) + o.z);
            r[4 * j + 3] = __float_as_uint(__uint_as_float(r[4 * j + 3]) + o.w);
          }
        }
        if (tma_out) {
          // Warp-uniform: this warp's 32 rows x 32 columns go out as one TMA box;
          // rows >= M and columns >= N are clipped by the tensor map.
          if (n0 + c0 < N && m0 + quarter * 32 < M) {
            uint8_t* box = my_out + (n_out & 1) * kOutBoxBytes;
            if (ep.kind == kEpiScaleMask) {
              // causal attention scores: key (column) after query (row) -> -inf
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const float val = (n0 + c0 + j > row) ? -INFINITY : ep.alpha * __uint_as_float(r[j]);
                r[j] = __float_as_uint(val);
              }
            }
            if (lane == 0) bulk_wait_read<1>();  // the box issued two rounds ago has been read
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const uint32_t off = lane * 128 + ((j ^ (lane & 7)) << 4);
              *reinterpret_cast<uint4*>(box + off) = make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              if constexpr (BATCHED) {
                tma_store_4d(&tmC, box, n0 + c0, m0 + quarter * 32, hb, sb);
              } else {
                if (ep.kind == kEpiF32Add)
                  tma_reduce_add_2d(&tmC, box, n0 + c0, m0 + quarter * 32, pol_out, hout != kL2None);
                else
                  tma_store_2d(&tmC, box, n0 + c0, m0 + quarter * 32, pol_out, hout != kL2None);
              }
              bulk_commit();
            }
            ++n_out;
          }
        } else if (n0 + c0 < N && m0 + quarter * 32 < M) {
          // Warp-uniform, as above: bf16 output box(es) of 32 rows x 32 columns.
          uint32_t o0[16], o1[16];
          const uint8_t* ib = nullptr;
          if (prefetch_in) {
            wait_in(n_in_used);
            ib = in_box(n_in_used++);
          }
          if constexpr (BATCHED) {
            if (ep.kind == kEpiSoftmaxGrad) {
              // dS = P (dP - delta) alpha, delta = sum_k P dP of this row (given)
              const float dl = row < M ? ep.g_in[(int64_t)(sb * nb_h + hb) * ep.ld + row] : 0.0f;
#pragma unroll
              for (int g = 0; g < 4; ++g) {
                float pv[8];
                ld_staged_bf16x8(ib, lane, g, pv);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                  o0[4 * g + j] = pack_bf16x2(pv[2 * j] * (__uint_as_float(r[8 * g + 2 * j]) - dl) * ep.alpha,
                                              pv[2 * j + 1] * (__uint_as_float(r[8 * g + 2 * j + 1]) - dl) * ep.alpha);
              }
            } else {
#pragma unroll
              for (int j = 0; j < 16; ++j)  // kEpiStore
                o0[j] = pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
            }
          } else {
            epilogue_dispatch(ep, row, n0 + c0, r, M, N, o0, o1, ib);
          }
          uint8_t* box0 = my_out + (n_out & 1) * (2 * kOutBoxBf16Bytes);
          uint8_t* box1 = box0 + kOutBoxBf16Bytes;
          const bool two = ep.kind == kEpiGelu;
          if (lane == 0) bulk_wait_read<1>();
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t off = lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4);
            *reinterpret_cast<uint4*>(box0 + off) = make_uint4(o0[4 * j], o0[4 * j + 1], o0[4 * j + 2], o0[4 * j + 3]);
            if (two)
              *reinterpret_cast<uint4*>(box1 + off) =
                  make_uint4(o1[4 * j], o1[4 * j + 1], o1[4 * j + 2], o1[4 * j + 3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if constexpr (BATCHED) {
              tma_store_4d(&tmO0, box0, n0 + c0, m0 + quarter * 32, hb, sb);
            } else {
              tma_store_2d(&tmO0, box0, n0 + c0, m0 + quarter * 32, pol_out, hout != kL2None);
              if (two) tma_store_2d(&tmO1, box1, n0 + c0, m0 + quarter * 32, pol_out, hout != kL2None);
            }
            bulk_commit();
          }
          ++n_out;
          // the input box just read is free again: refill it kInDepth blocks ahead
          // (the lanes' reads of it precede the fence and the warp barrier above)
          if (prefetch_in && ((c0 - col_begin) >> 5) + kInDepth < n_blocks)
            request_in(n0 + c0 + 32 * kInDepth, m0 + quarter * 32, hb, sb);
        }
      };
#pragma unroll 1
      for (int c0 = col_begin; c0 < (finisher ? col_end : col_begin); c0 += 32) {
        pace_block(c0);
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_row + c0, r);
        tmem_ld_wait();
        out_block(c0, r);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (PAIR)
          mbar_arrive_cluster(mapa_shared(smem_u32(&acc_empty[acc]), 0));
        else
          mbar_arrive(&acc_empty[acc]);
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
    if (lane == 0) bulk_wait_all();  // stores complete before the CTA (and its smem) goes away
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();  // the even CTA's MMAs no longer read the odd CTA's smem / TMEM
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<PAIR>(tmem_base, kTmemCols);
  }
  if (late_wait) grid_dependency_wait();
}

}  // namespace gbmlp
