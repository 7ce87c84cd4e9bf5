// C-ABI of the tensor-sliced MLP block: argument checks, TMA descriptors and the
// kernel sequence of the forward and backward passes on the caller's stream.
//
// Forward (per slice i, in turn):  F1  U_i, Y_i = GeLU(X A_i + a_i)        GEMM + GeLU epilogue
//                                  F2  Z += Y_i B_i; last slice: O = R + dropout(Z + b)
// Backward:                        B1  dZ = dropout'(dO), db (+)= sum dZ     element-wise + column sum
//                   (per slice)    B2  dU_i = (dZ B_i^T) * GeLU'(U_i)      GEMM + GeLU' epilogue
//                                      da_i (+)= sum dU_i                  column sum
//                                  B3  dB_i (+)= Y_i^T dZ                  GEMM + fp32 store / reduce-add
//                                  B4  dA_i (+)= X^T dU_i                  GEMM + fp32 store / reduce-add
// Weight and bias gradients are added to the fp32 accumulators, or, for the first
// micro-batch of a step (accumulate = 0), stored into them.
//                                  B5  dX (+)= dU_i A_i^T; last slice adds dO and writes bf16
// The forward sum over slices (operator g of the Megatron MLP) and the backward sum
// (operator f) are fp32 reductions in HBM on this GPU (STRONGHOLD slides, item 8).
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <utility>

#include <cuda.h>
#include <cuda_runtime.h>

#include "adam.cuh"
#include "attention.cuh"
#include "attn_fused.cuh"
#include "elementwise.cuh"
#include "gb_mlp.h"
#include "gemm_tc.cuh"

using namespace gbmlp;

namespace {

// Device status word: [0] = first error code, [1] = the site that recorded it.
__device__ int g_status_word[2];
// Partial sums and arrival counters of the GEMMs' split tail (static, so that no
// call allocates; the counters return to 0 after every use), one region per
// stream for up to kSplitRegions streams: launches on one stream never use the
// region at the same time (see gemm), launches on different streams may.
constexpr int kSplitRegions = 4;
__device__ float g_split_ws[kSplitRegions][kSplitSlots * 2 * kSplitSlotFloats];
__device__ int g_split_flags[kSplitRegions][kSplitSlots];
// Tile counters of the GEMMs' dynamic scheduler, one pair per stream region (the
// same regions as the split tail): both 0 between launches.
__device__ int g_sched_ctr[kSplitRegions][2];

thread_local std::string g_last_error;
std::atomic<uint64_t> g_launches{0};

// Optional per-launch timing: a CUDA event pair around every kernel launch.
struct TraceEntry {
  int kind;
  int64_t m, n, k;
};
struct TraceState {
  bool on = false;
  int capacity = 0;
  int count = 0;
  cudaEvent_t* ev = nullptr;  // 2 * capacity events
  TraceEntry* entries = nullptr;
};
std::mutex g_trace_mu;
TraceState g_trace;

// Kernel identifiers reported by the trace.
enum TraceKind {
  kTraceF1 = 0, kTraceF2 = 1, kTraceB2 = 2, kTraceB3 = 3, kTraceB4 = 4, kTraceB5 = 5,
  kTraceDropBwd = 10, kTraceColsum = 11, kTraceZero = 12, kTraceOther = 13, kTraceAdam = 14, kTraceTranspose = 15,
  kTraceAttnGemm = 20, kTraceSoftmax = 21, kTraceAttnCore = 22
};

// Records the start event of the next launch; returns its slot or -1.
int trace_pre(cudaStream_t s) {
  std::lock_guard<std::mutex> lock(g_trace_mu);
  if (!g_trace.on || g_trace.count >= g_trace.capacity) return -1;
  const int slot = g_trace.count++;
  cudaEventRecord(g_trace.ev[2 * slot], s);
  return slot;
}

void trace_post(int slot, cudaStream_t s, int kind, int64_t m, int64_t n, int64_t k) {
  if (slot < 0) return;
  std::lock_guard<std::mutex> lock(g_trace_mu);
  cudaEventRecord(g_trace.ev[2 * slot + 1], s);
  g_trace.entries[slot] = TraceEntry{kind, m, n, k};
}

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  int sms = 0;
  int* status = nullptr;
  float* split_ws = nullptr;   // partial sums of the GEMMs' split tail, kSplitRegions regions
  int* split_flags = nullptr;
  int* sched_ctr = nullptr;    // tile counters of the dynamic scheduler, 2 per region
  cudaStream_t split_owner[kSplitRegions] = {};  // the stream each region belongs to
  int split_regions_used = 0;
  bool gemm_attr[32] = {};  // per GEMM instantiation: dynamic smem attribute set
  bool fa_attr = false;     // fused attention core: dynamic smem attribute set
  bool fb_attr = false;     // fused attention backward core: dynamic smem attribute set
  int max_pairs[32] = {};   // per CTA-pair instantiation: co-resident clusters of two
};


std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Current device, checked to be sm_103; sets up per-device state once.
int device_state(DeviceState** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(MLP_EUNSUPPORTED, "no CUDA device: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(MLP_EUNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (major != 10 || minor != 3)
      return fail(MLP_EUNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a only", dev, major, minor);
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_status_word);
    if (e != cudaSuccess) return fail(MLP_ECUDA, "status word address: %s", cudaGetErrorString(e));
    void* ws = nullptr;
    void* flags = nullptr;
    void* ctr = nullptr;
    e = cudaGetSymbolAddress(&ws, g_split_ws);
    if (e == cudaSuccess) e = cudaGetSymbolAddress(&flags, g_split_flags);
    if (e == cudaSuccess) e = cudaGetSymbolAddress(&ctr, g_sched_ctr);
    if (e != cudaSuccess) return fail(MLP_ECUDA, "split-tail workspace address: %s", cudaGetErrorString(e));
    st.split_ws = static_cast<float*>(ws);
    st.split_flags = static_cast<int*>(flags);
    st.sched_ctr = static_cast<int*>(ctr);
    if (g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
        return fail(MLP_ECUDA, "cuTensorMapEncodeTiled unavailable");
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    st.sms = sms;
    st.status = static_cast<int*>(p);
    st.ready = true;
  }
  *out = &st;
  return MLP_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The region of `stream` (assigned on first use) in the static per-stream
// workspaces (split-tail partial sums, tile counters), or -1 once all regions
// belong to other streams; GEMMs on such a stream run without the split tail and
// with the static tile order.
std::mutex g_split_mu;
int split_region(DeviceState* st, cudaStream_t stream) {
  std::lock_guard<std::mutex> lock(g_split_mu);
  for (int r = 0; r < st->split_regions_used; ++r)
    if (st->split_owner[r] == stream) return r;
  if (st->split_regions_used == kSplitRegions) return -1;
  st->split_owner[st->split_regions_used] = stream;
  return st->split_regions_used++;
}

// Programmatic dependent launch: a kernel may be scheduled while the previous
// kernel on its stream drains, running its prologue (barriers, TMEM, descriptor
// prefetch) early; every kernel of this library executes griddepcontrol.wait
// before its first global-memory access, so results are unchanged.  On by default.
std::atomic<int> g_pdl{1};

// Launch through cudaLaunchKernelEx with an optional (cx, cy, 1) cluster and the
// programmatic-serialization attribute.
template <typename... Params, typename... Args>
cudaError_t launch_kernel(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, unsigned cx,
                          unsigned cy, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (cx * cy > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cx;
    attr[n].val.clusterDim.y = cy;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (g_pdl.load(std::memory_order_relaxed)) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

#include "gemm_host.cuh"

DropoutParams make_dropout(float p, uint64_t seed, uint64_t token_offset, int h) {
  DropoutParams d;
  d.seed = seed;
  d.token_offset = token_offset;
  d.row_width = (uint64_t)h;
  d.thr = (uint64_t)llround((double)p * 4294967296.0);
  d.scale = 1.0f / (1.0f - p);
  return d;
}

int check_shape(int h, int ffn, int t, int slice, int64_t tokens, float p) {
  if (h <= 0 || h % 8 != 0) return fail(MLP_EINVAL, "h = %d must be positive and a multiple of 8", h);
  if (t <= 0 || ffn <= 0 || ffn % t != 0) return fail(MLP_EINVAL, "ffn = %d must be a positive multiple of t = %d", ffn, t);
  if ((ffn / t) % 8 != 0) return fail(MLP_EINVAL, "f = ffn / t = %d must be a multiple of 8", ffn / t);
  if (tokens <= 0 || tokens >= (int64_t)1 << 31) return fail(MLP_EINVAL, "tokens = %lld out of range", (long long)tokens);
  if (!(p >= 0.0f && p < 1.0f)) return fail(MLP_EINVAL, "dropout probability p = %g not in [0, 1)", (double)p);
  if (slice < -1 || slice >= t) return fail(MLP_EINVAL, "slice = %d not in [-1, t = %d)", slice, t);
  return MLP_OK;
}

int check_ptrs(const char* what, std::initializer_list<const void*> ptrs) {
  int idx = 0;
  for (const void* p : ptrs) {
    if (p == nullptr) return fail(MLP_EINVAL, "%s: pointer argument %d is NULL", what, idx);
    if (!aligned16(p)) return fail(MLP_EALIGN, "%s: pointer argument %d is not 16-byte aligned", what, idx);
    ++idx;
  }
  return MLP_OK;
}

// CTAs per column block of the (memory-bound) column sum: the most (1, 2, 4 or 8)
// for which the whole grid is resident at once (a second, partial wave would take
// as long as the first); the choice depends on the shape and the device only, so
// the summation order, and the result, is fixed for a shape.
template <typename Kernel>
unsigned colsum_split(const DeviceState* st, int64_t cols, Kernel kernel) {
  static int per_sm = 0;  // per kernel (each kernel has its own signature, hence instantiation)
  if (per_sm == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kColThreads, 0) != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = 1;
    }
    per_sm = n;
  }
  const int64_t blocks = (cols + kColsPerCta - 1) / kColsPerCta;
  const int64_t resident = (int64_t)per_sm * st->sms;
  unsigned split = 1;
  while (split < (unsigned)kColRowSplitMax && blocks * split * 2 <= resident) split *= 2;
  return split;
}

// CTAs per column block of the dropout backward, whose mask hashing makes it
// arithmetic-bound: the fewest (1, 2, 4 or 8) that give at least four CTAs per SM
// (measured on the MT-NLG layer: 114 us with one wave of 320 CTAs, 99 us with 640).
unsigned dropout_bwd_split(const DeviceState* st, int64_t cols) {
  const int64_t blocks = (cols + kColsPerCta - 1) / kColsPerCta;
  unsigned split = 1;
  while (split < (unsigned)kColRowSplitMax && blocks * split < 4 * (int64_t)st->sms) split *= 2;
  return split;
}

// Transposed operands for the weight-gradient GEMMs (mlp_set_wgrad_transpose).
std::atomic<int> g_wgrad_transpose{-1};
// Below this size per GEMM the copies cost more than they save (the mid workload's
// 0.27 TFLOP weight-gradient GEMMs: 6 us saved, 14 us of copies).
constexpr double kWgradTransposeMinFlop = 1e12;

// Whether a weight-gradient GEMM D[M, N] (+)= A^T B, reducing over T tokens, may
// read a transposed copy of one operand as a K-major operand: the switch allows
// it, the scratch for the copy is there and 16-byte aligned, the token count
// suits the copy kernel and the tensor maps (a multiple of 8), and the GEMM takes
// the CTA-pair form with a reduction of 16 k-blocks or more (the forms the
// (K, MN) and (MN, K) launches instantiate); by default, only GEMMs large enough
// to repay the copy.
bool wgrad_transposed(int M, int N, int64_t T, const void* scratch) {
  const int mode = g_wgrad_transpose.load(std::memory_order_relaxed);
  if (mode == 0 || scratch == nullptr || (reinterpret_cast<uintptr_t>(scratch) & 15) != 0) return false;
  if (T % 8 != 0 || (T + kTrTile - 1) / kTrTile > 65535) return false;
  const int pm = g_pair_mode.load(std::memory_order_relaxed);
  if (pm == 0 || (pm < 0 && M <= kBM) || (T + kBK - 1) / kBK < 16) return false;
  return mode == 1 || 2.0 * (double)M * (double)N * (double)T >= kWgradTransposeMinFlop;
}

int launch_check(cudaError_t e, const char* what) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return fail(MLP_ECUDA, "%s launch: %s", what, cudaGetErrorString(e));
  return MLP_OK;
}

// One launch of k_transpose_bf16 for one or two [rows, cols] matrices (j1.in may
// be null), traced as kTraceTranspose.
int launch_transposes(cudaStream_t s, int64_t rows, int cols, TransposeJob j0, TransposeJob j1, const char* what) {
  const unsigned jobs = j1.in != nullptr ? 2u : 1u;
  const int ts = trace_pre(s);
  const cudaError_t e = launch_kernel(k_transpose_bf16, dim3((cols + kTrTile - 1) / kTrTile,
                                                             (unsigned)((rows + kTrTile - 1) / kTrTile), jobs),
                                      dim3(kTrThreads), 0, s, 1, 1, j0, j1, rows, cols);
  trace_post(ts, s, kTraceTranspose, rows, cols, 0);
  return launch_check(e, what);
}

template <int CHUNKS>
cudaError_t softmax_warp_launch(DeviceState* st, const float* S, uint16_t* P, int64_t rows, int cols, cudaStream_t s) {
  const int64_t ctas_needed = (rows + kSoftmaxRowsPerCta - 1) / kSoftmaxRowsPerCta;
  const int64_t blocks = ctas_needed < (int64_t)st->sms * 8 ? ctas_needed : (int64_t)st->sms * 8;
  return launch_kernel(k_softmax_rows_warp<CHUNKS>, dim3((unsigned)blocks), dim3(kSoftmaxRowsPerCta * 32), 0, s, 1, 1,
                       S, P, rows, cols);
}

}  // namespace

namespace gbmlp {
void set_last_error(const char* msg) { g_last_error = msg; }
}  // namespace gbmlp

extern "C" {

int mlp_fwd(int h, int ffn, int t, int slice, int64_t tokens, float p, uint64_t seed, uint64_t token_offset,
            const mlp_bf16* X, const mlp_bf16* A, const mlp_bf16* a, const mlp_bf16* B, const mlp_bf16* b,
            const mlp_bf16* R, mlp_bf16* U, mlp_bf16* Y, float* Zacc, mlp_bf16* O, void* stream) {
  int rc = check_shape(h, ffn, t, slice, tokens, p);
  if (rc) return rc;
  rc = check_ptrs("mlp_fwd", {X, A, a, B, b, U, Y, O});
  if (rc) return rc;
  if (R != nullptr && !aligned16(R)) return fail(MLP_EALIGN, "mlp_fwd: R is not 16-byte aligned");
  if (t > 1 && slice >= 0) {
    rc = check_ptrs("mlp_fwd (Zacc, needed for one-slice calls when t > 1)", {Zacc});
    if (rc) return rc;
  }
  DeviceState* st = nullptr;
  rc = device_state(&st);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int T = (int)tokens;
  const DropoutParams drop = make_dropout(p, seed, token_offset, h);
  if (R == nullptr) R = X;
  // All slices in one call: each GEMM launch covers every slice.  F1 walks the
  // column blocks A_0 .. A_{t-1} tile by tile, and F2's reduction loop walks the
  // row blocks B_0 .. B_{t-1}, so the sum over slices of the partial products
  // Y_i B_i happens in the TMEM accumulator.  One-slice calls reduce through Zacc.
  if (slice < 0) t = 1;
  const int f = ffn / t;
  const int i0 = slice < 0 ? 0 : slice;
  const int i1 = slice < 0 ? 1 : slice + 1;
  for (int i = i0; i < i1; ++i) {
    // F1: U_i = X A_i + a_i, Y_i = GeLU(U_i)          (M = T, N = f, K = h)
    EpiParams e1{};
    e1.kind = kEpiGelu;
    e1.ld = ffn;
    e1.out0 = U + (int64_t)i * f;
    e1.out1 = Y + (int64_t)i * f;
    e1.bias = a + (int64_t)i * f;
    rc = gemm(st, X, false, h, A + (int64_t)i * f, true, ffn, T, f, h, e1, s, kTraceF1);
    if (rc) return rc;
    // F2: Z (+)= Y_i B_i; the last slice finishes O = R + dropout(Z + b)   (M = T, N = h, K = f)
    EpiParams e2{};
    e2.ld = h;
    if (t == 1 || i == t - 1) {
      e2.kind = kEpiDropRes;
      e2.g_in = (t == 1) ? nullptr : Zacc;
      e2.in0 = R;
      e2.bias = b;
      e2.out0 = O;
      e2.drop = drop;
    } else {
      e2.kind = (i == 0) ? kEpiF32Store : kEpiF32Add;
      e2.g_out = Zacc;
    }
    rc = gemm(st, Y + (int64_t)i * f, false, ffn, B + (int64_t)i * f * h, true, h, T, h, f, e2, s, kTraceF2);
    if (rc) return rc;
  }
  return MLP_OK;
}

int mlp_bwd(int h, int ffn, int t, int slice, int64_t tokens, float p, uint64_t seed, uint64_t token_offset,
            int residual_grad, int accumulate, const mlp_bf16* dO, const mlp_bf16* X, const mlp_bf16* A, const mlp_bf16* B,
            const mlp_bf16* U, const mlp_bf16* Y, mlp_bf16* dZ, mlp_bf16* dU, float* dXacc, mlp_bf16* dX,
            float* dA, float* da, float* dB, float* db, void* stream) {
  int rc = check_shape(h, ffn, t, slice, tokens, p);
  if (rc) return rc;
  rc = check_ptrs("mlp_bwd", {dO, X, A, B, U, Y, dZ, dU, dX, dA, da, dB, db});
  if (rc) return rc;
  if (t > 1 && slice >= 0) {
    rc = check_ptrs("mlp_bwd (dXacc, needed for one-slice calls when t > 1)", {dXacc});
    if (rc) return rc;
  }
  DeviceState* st = nullptr;
  rc = device_state(&st);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int T = (int)tokens;
  const DropoutParams drop = make_dropout(p, seed, token_offset, h);
  const bool first_call = slice <= 0;
  // All slices in one call: B2, B3, B4 cover every slice's columns in one launch
  // each, and B5's reduction loop walks A_0^T .. A_{t-1}^T so the sum over slices
  // of dU_i A_i^T happens in the TMEM accumulator.  One-slice calls use dXacc.
  if (slice < 0) t = 1;
  const int f = ffn / t;
  if (first_call) {
    // B1: dZ = dO * m / (1 - p), db += sum_tok dZ
    const int ts = trace_pre(s);
    const unsigned split = dropout_bwd_split(st, h);
    const cudaError_t e = launch_kernel(k_dropout_bwd_colsum, dim3((h + kColsPerCta - 1) / kColsPerCta, split),
                                        dim3(kColThreads), 0, s, 1, split, dO, dZ, db, tokens, h, drop,
                                        accumulate ? 1 : 0);
    trace_post(ts, s, kTraceDropBwd, tokens, h, 0);
    rc = launch_check(e, "dropout backward");
    if (rc) return rc;
  }
  // B3 and B4 reduce over the tokens, so both of their operands are MN-major as
  // stored, and a GEMM with two MN-major operands runs about 5 % slower than one
  // with a K-major operand (measured on the MT-NLG layer).  When dXacc is free (t == 1
  // or the all-slices call) and the GEMMs are large, it holds transposed copies X^T
  // and dZ^T ([h, tokens] bf16 each: together exactly dXacc's bytes), made by one
  // launch after B1; B3 reads dZ^T and B4 X^T as K-major operands.  Same products,
  // same reduction order per tile.
  mlp_bf16* Xt = nullptr;
  mlp_bf16* dZt = nullptr;
  if (t == 1 && wgrad_transposed(f, h, tokens, dXacc) && wgrad_transposed(h, f, tokens, dXacc)) {
    Xt = reinterpret_cast<mlp_bf16*>(dXacc);
    dZt = Xt + (int64_t)h * tokens;
    rc = launch_transposes(s, tokens, h, TransposeJob{X, Xt}, TransposeJob{dZ, dZt}, "transposed copies of X and dZ");
    if (rc) return rc;
  }
  const int i0 = slice < 0 ? 0 : slice;
  const int i1 = slice < 0 ? 1 : slice + 1;
  for (int i = i0; i < i1; ++i) {
    const int64_t c = (int64_t)i * f;
    // B2: dU_i = (dZ B_i^T) * GeLU'(U_i)                 (M = T, N = f, K = h)
    EpiParams e2{};
    e2.kind = kEpiDGelu;
    e2.ld = ffn;
    e2.in0 = U + c;
    e2.out0 = dU + c;
    rc = gemm(st, dZ, false, h, B + c * h, false, h, T, f, h, e2, s, kTraceB2);
    if (rc) return rc;
    // da_i += sum_tok dU_i
    const int ts = trace_pre(s);
    const unsigned split = colsum_split(st, f, k_colsum_bf16);
    const cudaError_t e = launch_kernel(k_colsum_bf16, dim3((f + kColsPerCta - 1) / kColsPerCta, split),
                                        dim3(kColThreads), 0, s, 1, split, (const uint16_t*)(dU + c),
                                        (int64_t)ffn, da + c, tokens, f, accumulate ? 1 : 0);
    trace_post(ts, s, kTraceColsum, tokens, f, 0);
    rc = launch_check(e, "bias-gradient column sum");
    if (rc) return rc;
    // B5, B3 and B4 read only dU (B2), dZ (B1) and the forward's tensors, so each
    // may start while its predecessor drains (late dependency wait); B5 goes
    // first, so that B3's tiles fill B5's last, partial wave.
    // B5: dX (+)= dU_i A_i^T; the last slice adds dO and writes bf16   (M = T, N = h, K = f)
    EpiParams e5{};
    e5.ld = h;
    if (t == 1 || i == t - 1) {
      e5.kind = kEpiResAdd;
      e5.g_in = (t == 1) ? nullptr : dXacc;
      e5.in0 = residual_grad ? dO : nullptr;
      e5.out0 = dX;
    } else {
      e5.kind = (i == 0) ? kEpiF32Store : kEpiF32Add;
      e5.g_out = dXacc;
    }
    rc = gemm(st, dU + c, false, ffn, A + c, false, ffn, T, h, f, e5, s, kTraceB5, true);
    if (rc) return rc;
    // B3: dB_i (+)= Y_i^T dZ                             (M = f, N = h, K = T)
    EpiParams e3{};
    e3.kind = accumulate ? kEpiF32Add : kEpiF32Store;
    e3.ld = h;
    e3.g_out = dB + c * h;
    rc = dZt ? gemm(st, Y + c, true, ffn, dZt, false, T, f, h, T, e3, s, kTraceB3, true)
             : gemm(st, Y + c, true, ffn, dZ, true, h, f, h, T, e3, s, kTraceB3, true);
    if (rc) return rc;
    // B4: dA_i (+)= X^T dU_i                             (M = h, N = f, K = T)
    EpiParams e4{};
    e4.kind = accumulate ? kEpiF32Add : kEpiF32Store;
    e4.ld = ffn;
    e4.g_out = dA + c;
    rc = Xt ? gemm(st, Xt, false, T, dU + c, true, ffn, h, f, T, e4, s, kTraceB4, true)
            : gemm(st, X, true, h, dU + c, true, ffn, h, f, T, e4, s, kTraceB4, true);
    if (rc) return rc;
  }
  return MLP_OK;
}

int grad_accum_reset(int h, int ffn, float* dA, float* da, float* dB, float* db, void* stream) {
  if (h <= 0 || h % 8 != 0 || ffn <= 0 || ffn % 8 != 0)
    return fail(MLP_EINVAL, "grad_accum_reset: h = %d and ffn = %d must be positive multiples of 8", h, ffn);
  int rc = check_ptrs("grad_accum_reset", {dA, da, dB, db});
  if (rc) return rc;
  DeviceState* st = nullptr;
  rc = device_state(&st);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* bufs[4] = {dA, da, dB, db};
  const int64_t sizes[4] = {(int64_t)h * ffn, ffn, (int64_t)ffn * h, h};
  for (int k = 0; k < 4; ++k) {
    const int64_t n4 = sizes[k] / 4;
    int64_t blocks = (n4 + 255) / 256;
    if (blocks > (int64_t)st->sms * 8) blocks = (int64_t)st->sms * 8;
    if (blocks < 1) blocks = 1;
    const int ts = trace_pre(s);
    const cudaError_t e = launch_kernel(k_zero_f32, dim3((unsigned)blocks), dim3(256), 0, s, 1, 1, bufs[k], sizes[k]);
    trace_post(ts, s, kTraceZero, sizes[k], 0, 0);
    rc = launch_check(e, "grad_accum_reset");
    if (rc) return rc;
  }
  return MLP_OK;
}

int check_attn_shape(int h, int nh, int t, int64_t tokens, int seq_len, float p) {
  if (h <= 0 || h % 8 != 0) return fail(MLP_EINVAL, "attention: h = %d must be a positive multiple of 8", h);
  if (nh <= 0 || h % nh != 0 || (h / nh) % 8 != 0)
    return fail(MLP_EINVAL, "attention: head size h / nh must be a whole multiple of 8 (h %d, nh %d)", h, nh);
  if (t <= 0 || nh % t != 0) return fail(MLP_EINVAL, "attention: nh = %d must be a multiple of t = %d", nh, t);
  if (seq_len <= 0 || seq_len % 8 != 0) return fail(MLP_EINVAL, "attention: seq_len = %d must be a multiple of 8", seq_len);
  if (tokens <= 0 || tokens >= (int64_t)1 << 31 || tokens % seq_len != 0)
    return fail(MLP_EINVAL, "attention: tokens = %lld must be a positive multiple of seq_len", (long long)tokens);
  if (!(p >= 0.0f && p < 1.0f)) return fail(MLP_EINVAL, "attention: dropout p = %g not in [0, 1)", (double)p);
  return MLP_OK;
}

// 1 (the default): the attention forward's core (S = Q K^T, softmax, O = P V) runs
// as one fused kernel when the head size is at most 192; 0: three launches with S
// in HBM (a batched GEMM, the row softmax, a batched GEMM).
std::atomic<int> g_attn_fused{1};

// The fused attention core over every (sequence, head, query tile); P and O as in
// attn_fwd.  Returns MLP_OK or an error code.
int attn_core_fused(DeviceState* st, const uint16_t* QKV, uint16_t* P, uint16_t* O, int h, int nh, int L, int ns,
                    cudaStream_t s) {
  const int d = h / nh;
  const int64_t h3 = 3 * (int64_t)h;
  FaParams fp;
  fp.L = L;
  fp.nh = nh;
  fp.ns = ns;
  fp.d = d;
  fp.d_pad = (d + 15) & ~15;
  fp.n_atoms = (fp.d_pad + 63) / 64;
  fp.alpha = 1.0f / std::sqrt((float)d);
  fp.P = P;
  CUtensorMap mQ, mK, mV, mP, mO;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  int rc = make_map4(&mQ, bf, 2, QKV, d, L, h3, nh, d, ns, L * h3, 64, kFaTile, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  if (!rc)
    rc = make_map4(&mK, bf, 2, QKV + h, d, L, h3, nh, d, ns, L * h3, 64, kFaTile, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  if (!rc)
    rc = make_map4(&mV, bf, 2, QKV + 2 * h, d, L, h3, nh, d, ns, L * h3, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  if (!rc)
    rc = make_map4(&mP, bf, 2, P, L, L, L, nh, (int64_t)L * L, ns, (int64_t)nh * L * L, 64, 32,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE);
  if (!rc)
    rc = make_map4(&mO, bf, 2, O, d, L, h, nh, d, ns, (int64_t)L * h, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE);
  if (rc) return rc;
  if (!st->fa_attr) {
    const cudaError_t e =
        cudaFuncSetAttribute(k_attn_fwd_fused, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFaSmemBytes);
    if (e != cudaSuccess) return fail(MLP_ECUDA, "cudaFuncSetAttribute (fused attention): %s", cudaGetErrorString(e));
    st->fa_attr = true;
  }
  const int64_t items = (int64_t)((L + kFaTile - 1) / kFaTile) * nh * ns;
  const unsigned grid = (unsigned)(items < st->sms ? items : st->sms);
  const int ts = trace_pre(s);
  const cudaError_t e = launch_kernel(k_attn_fwd_fused, dim3(grid), dim3(kFaThreads), kFaSmemBytes, s, 1, 1, mQ, mK,
                                      mV, mP, mO, fp, st->status);
  trace_post(ts, s, kTraceAttnCore, (int64_t)ns * nh * L, L, d);
  return launch_check(e, "fused attention core");
}

// The fused attention core of the backward: dK and dV into dQKV, dS (P's shape)
// into dS; delta = rowsum(dO * O) must be in `delta`.
int attn_core_bwd_fused(DeviceState* st, const uint16_t* QKV, const uint16_t* P, const uint16_t* dO,
                        const float* delta, uint16_t* dS, uint16_t* dQKV, int h, int nh, int L, int ns,
                        cudaStream_t s) {
  const int d = h / nh;
  const int64_t h3 = 3 * (int64_t)h, LL = (int64_t)L * L;
  FbParams fb;
  fb.L = L;
  fb.nh = nh;
  fb.ns = ns;
  fb.d = d;
  fb.d_pad = (d + 15) & ~15;
  fb.n_atoms = (fb.d_pad + 63) / 64;
  fb.alpha = 1.0f / std::sqrt((float)d);
  fb.dS = dS;
  CUtensorMap mV, mQ, mdO, mP, mDelta, mDS, mdK, mdV;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto sw128 = CU_TENSOR_MAP_SWIZZLE_128B;
  const auto l2 = CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
  int rc = make_map4(&mV, bf, 2, QKV + 2 * h, d, L, h3, nh, d, ns, L * h3, 64, kFaTile, sw128, l2);
  if (!rc) rc = make_map4(&mQ, bf, 2, QKV, d, L, h3, nh, d, ns, L * h3, 64, kFaTile, sw128, l2);
  if (!rc) rc = make_map4(&mdO, bf, 2, dO, d, L, h, nh, d, ns, (int64_t)L * h, 64, kFaTile, sw128, l2);
  if (!rc) rc = make_map4(&mP, bf, 2, P, L, L, L, nh, LL, ns, nh * LL, 64, kFaTile, sw128, l2);
  if (!rc)
    rc = make_map4(&mDS, bf, 2, dS, L, L, L, nh, LL, ns, nh * LL, 64, 32, sw128, CU_TENSOR_MAP_L2_PROMOTION_NONE);
  if (!rc)
    rc = make_map4(&mdK, bf, 2, dQKV + h, d, L, h3, nh, d, ns, L * h3, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE);
  if (!rc)
    rc = make_map4(&mdV, bf, 2, dQKV + 2 * h, d, L, h3, nh, d, ns, L * h3, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE);
  if (rc) return rc;
  {
    // delta: fp32 [ns * nh rows][L], one 128-query box per load (zero past L)
    cuuint64_t dims[2] = {(cuuint64_t)L, (cuuint64_t)ns * nh};
    cuuint64_t strides[1] = {(cuuint64_t)L * 4};
    cuuint32_t box[2] = {(cuuint32_t)kFaTile, 1};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(&mDelta, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(delta), dims, strides,
                                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MLP_ECUDA, "cuTensorMapEncodeTiled (softmax-gradient row sums) failed (%d)", (int)r);
  }
  if (!st->fb_attr) {
    const cudaError_t e =
        cudaFuncSetAttribute(k_attn_bwd_fused, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFbSmemBytes);
    if (e != cudaSuccess)
      return fail(MLP_ECUDA, "cudaFuncSetAttribute (fused attention backward): %s", cudaGetErrorString(e));
    st->fb_attr = true;
  }
  const int64_t items = (int64_t)((L + kFaTile - 1) / kFaTile) * nh * ns;
  const unsigned grid = (unsigned)(items < st->sms ? items : st->sms);
  const int ts = trace_pre(s);
  const cudaError_t e = launch_kernel(k_attn_bwd_fused, dim3(grid), dim3(kFbThreads), kFbSmemBytes, s, 1, 1, mV, mQ,
                                      mdO, mP, mDelta, mDS, mdK, mdV, fb, st->status);
  trace_post(ts, s, kTraceAttnCore, (int64_t)ns * nh * L, L, d);
  return launch_check(e, "fused attention backward core");
}

int softmax_launch(DeviceState* st, const float* S, uint16_t* P, int64_t rows, int cols, cudaStream_t s) {
  int64_t blocks = rows < (int64_t)st->sms * 16 ? rows : (int64_t)st->sms * 16;
  const int ts = trace_pre(s);
  const int chunks = (cols + 255) / 256;
  const cudaError_t e =
      chunks <= 1   ? softmax_warp_launch<1>(st, S, P, rows, cols, s)
      : chunks <= 2 ? softmax_warp_launch<2>(st, S, P, rows, cols, s)
      : chunks <= 4 ? softmax_warp_launch<4>(st, S, P, rows, cols, s)
      : chunks <= 8 ? softmax_warp_launch<8>(st, S, P, rows, cols, s)
                    : launch_kernel(k_softmax_rows, dim3((unsigned)blocks), dim3(kSoftmaxThreads), 0, s, 1, 1, S, P,
                                    rows, cols);
  trace_post(ts, s, kTraceSoftmax, rows, cols, 0);
  return launch_check(e, "softmax");
}

int adam_step(int64_t n, const float* grad, float grad_scale, float* master, float* m, float* v, mlp_bf16* weight,
              float lr, float beta1, float beta2, float eps, float weight_decay, int step, void* stream) {
  if (n <= 0) return fail(MLP_EINVAL, "adam_step: n = %lld must be positive", (long long)n);
  if (step < 1) return fail(MLP_EINVAL, "adam_step: step = %d must be >= 1", step);
  if (!(beta1 >= 0.0f && beta1 < 1.0f && beta2 >= 0.0f && beta2 < 1.0f))
    return fail(MLP_EINVAL, "adam_step: betas (%g, %g) not in [0, 1)", (double)beta1, (double)beta2);
  if (!(eps > 0.0f) || !(lr >= 0.0f) || !(weight_decay >= 0.0f))
    return fail(MLP_EINVAL, "adam_step: eps must be > 0, lr and weight_decay >= 0");
  int rc = check_ptrs("adam_step", {grad, master, m, v});
  if (rc) return rc;
  if (weight == nullptr || (reinterpret_cast<uintptr_t>(weight) & 7u) != 0)
    return fail(weight == nullptr ? MLP_EINVAL : MLP_EALIGN, "adam_step: weight NULL or not 8-byte aligned");
  DeviceState* st = nullptr;
  rc = device_state(&st);
  if (rc) return rc;
  AdamParams p;
  p.grad_scale = grad_scale;
  p.beta1 = beta1;
  p.one_minus_beta1 = 1.0f - beta1;
  p.beta2 = beta2;
  p.one_minus_beta2 = 1.0f - beta2;
  const double bc1 = 1.0 - std::pow((double)beta1, step);
  const double bc2 = 1.0 - std::pow((double)beta2, step);
  p.step_size = (float)((double)lr / bc1);
  p.inv_sqrt_bc2 = (float)(1.0 / std::sqrt(bc2));
  p.eps = eps;
  p.decay = (float)(1.0 - (double)lr * (double)weight_decay);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int64_t blocks = (n / 4 + 255) / 256;
  if (blocks > (int64_t)st->sms * 8) blocks = (int64_t)st->sms * 8;
  if (blocks < 1) blocks = 1;
  const int ts = trace_pre(s);
  const cudaError_t e =
      launch_kernel(k_adam_step, dim3((unsigned)blocks), dim3(256), 0, s, 1, 1, n, grad, master, m, v, weight, p);
  trace_post(ts, s, kTraceAdam, n, 0, 0);
  return launch_check(e, "adam_step");
}

int attn_fwd(int h, int nh, int t, int64_t tokens, int seq_len, float p, uint64_t seed, uint64_t token_offset,
             const mlp_bf16* X, const mlp_bf16* Wqkv, const mlp_bf16* bqkv, const mlp_bf16* Wo, const mlp_bf16* bo,
             const mlp_bf16* R, mlp_bf16* QKV, float* S, mlp_bf16* P, mlp_bf16* O, mlp_bf16* out, void* stream) {
  int rc = check_attn_shape(h, nh, t, tokens, seq_len, p);
  if (rc) return rc;
  rc = check_ptrs("attn_fwd", {X, Wqkv, bqkv, Wo, bo, QKV, S, P, O, out});
  if (rc) return rc;
  if (R != nullptr && !aligned16(R)) return fail(MLP_EALIGN, "attn_fwd: R is not 16-byte aligned");
  DeviceState* st = nullptr;
  rc = device_state(&st);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (R == nullptr) R = X;
  const int T = (int)tokens, d = h / nh, L = seq_len, ns = T / L;
  const int64_t h3 = 3 * (int64_t)h, LL = (int64_t)L * L;
  // QKV = X Wqkv + bqkv: every slice's heads in one launch (column split of Wqkv)
  EpiParams e{};
  e.kind = kEpiBias;
  e.ld = h3;
  e.out0 = QKV;
  e.bias = bqkv;
  rc = gemm(st, X, false, h, Wqkv, true, h3, T, (int)h3, h, e, s, kTraceAttnGemm);
  if (rc) return rc;
  if (g_attn_fused.load(std::memory_order_relaxed) && ((d + 15) & ~15) <= kFaMaxAtoms * 64) {
    // S = Q K^T / sqrt(d), P = softmax(S), O = P V in one kernel; S stays on chip
    rc = attn_core_fused(st, QKV, P, O, h, nh, L, ns, s);
    if (rc) return rc;
    EpiParams ezf{};
    ezf.kind = kEpiDropRes;
    ezf.ld = h;
    ezf.in0 = R;
    ezf.bias = bo;
    ezf.out0 = out;
    ezf.drop = make_dropout(p, seed, token_offset, h);
    return gemm(st, O, false, h, Wo, true, h, T, h, h, ezf, s, kTraceAttnGemm);
  }
  // S = Q K^T / sqrt(d), -inf above the diagonal; per (sequence, head)
  EpiParams es{};
  es.kind = kEpiScaleMask;
  es.alpha = 1.0f / std::sqrt((float)d);
  rc = gemm_batched(st, {QKV, false, L, d, h3, d, L * h3}, {QKV + h, false, L, d, h3, d, L * h3},
                    {S, L, L, L, LL, nh * LL}, L, L, d, nh, ns, es, s, kTraceAttnGemm, kCausalSkipUpper);
  if (rc) return rc;
  rc = softmax_launch(st, S, P, (int64_t)ns * nh * L, L, s);
  if (rc) return rc;
  // O = P V per head, written into head j's columns of O
  EpiParams eo{};
  eo.kind = kEpiStore;
  rc = gemm_batched(st, {P, false, L, L, L, LL, nh * LL}, {QKV + 2 * h, true, d, L, h3, d, L * h3},
                    {O, d, L, h, d, (int64_t)L * h}, L, d, L, nh, ns, eo, s, kTraceAttnGemm, kCausalKUpTo);
  if (rc) return rc;
  // out = R + dropout(O Wo + bo): the row split of Wo summed over slices in the accumulator
  EpiParams ez{};
  ez.kind = kEpiDropRes;
  ez.ld = h;
  ez.in0 = R;
  ez.bias = bo;
  ez.out0 = out;
  ez.drop = make_dropout(p, seed, token_offset, h);
  return gemm(st, O, false, h, Wo, true, h, T, h, h, ez, s, kTraceAttnGemm);
}

int attn_bwd(int h, int nh, int t, int64_t tokens, int seq_len, float p, uint64_t seed, uint64_t token_offset,
             int residual_grad, int accumulate, const mlp_bf16* dOut, const mlp_bf16* X, const mlp_bf16* Wqkv,
             const mlp_bf16* Wo, const mlp_bf16* QKV, const mlp_bf16* P, const mlp_bf16* O, mlp_bf16* dZ,
             mlp_bf16* dO, float* dP, mlp_bf16* dS, mlp_bf16* dQKV, mlp_bf16* dX, float* dWqkv, float* dbqkv,
             float* dWo, float* dbo, void* stream) {
  int rc = check_attn_shape(h, nh, t, tokens, seq_len, p);
  if (rc) return rc;
  rc = check_ptrs("attn_bwd", {dOut, X, Wqkv, Wo, QKV, P, O, dZ, dO, dP, dS, dQKV, dX, dWqkv, dbqkv, dWo, dbo});
  if (rc) return rc;
  DeviceState* st = nullptr;
  rc = device_state(&st);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int T = (int)tokens, d = h / nh, L = seq_len, ns = T / L;
  const int64_t h3 = 3 * (int64_t)h, LL = (int64_t)L * L;
  const int acc = accumulate ? 1 : 0;
  // dZ = dropout'(dOut), dbo (+)= sum dZ
  {
    const DropoutParams drop = make_dropout(p, seed, token_offset, h);
    const int ts = trace_pre(s);
    const unsigned split = dropout_bwd_split(st, h);
    const cudaError_t e = launch_kernel(k_dropout_bwd_colsum, dim3((h + kColsPerCta - 1) / kColsPerCta, split),
                                        dim3(kColThreads), 0, s, 1, split, dOut, dZ, dbo, tokens, h, drop, acc);
    trace_post(ts, s, kTraceDropBwd, tokens, h, 0);
    rc = launch_check(e, "dropout backward");
    if (rc) return rc;
  }
  // dWo (+)= O^T dZ.  Both operands are MN-major as stored (the reduction runs over
  // the tokens); as for mlp_bwd's B3, a large enough GEMM reads a transposed copy
  // dZ^T instead, held in the dS workspace, which is free until the attention core
  // writes it (dS holds ns nh L L >= tokens h elements when L >= d).
  const bool ds_holds_copy = L >= d;
  EpiParams ew{};
  ew.kind = acc ? kEpiF32Add : kEpiF32Store;
  ew.ld = h;
  ew.g_out = dWo;
  if (ds_holds_copy && wgrad_transposed(h, h, tokens, dS)) {
    rc = launch_transposes(s, tokens, h, TransposeJob{dZ, dS}, TransposeJob{nullptr, nullptr}, "transposed copy of dZ");
    if (rc) return rc;
    rc = gemm(st, O, true, h, dS, false, T, h, h, T, ew, s, kTraceAttnGemm);
  } else {
    rc = gemm(st, O, true, h, dZ, true, h, h, h, T, ew, s, kTraceAttnGemm);
  }
  if (rc) return rc;
  // dO = dZ Wo^T
  EpiParams ed{};
  ed.kind = kEpiStore;
  ed.ld = h;
  ed.out0 = dO;
  rc = gemm(st, dZ, false, h, Wo, false, h, T, h, h, ed, s, kTraceAttnGemm);
  if (rc) return rc;
  EpiParams est{};
  est.kind = kEpiStore;
  if (g_attn_fused.load(std::memory_order_relaxed) && ((d + 15) & ~15) <= kFaMaxAtoms * 64) {
    // delta = rowsum(dO * O); then, fused per (sequence, head, key tile): dV, dK and
    // dS, and dQ = dS K as a batched GEMM
    float* delta = dP;
    {
      const int64_t warps = tokens * nh;
      int64_t blocks = (warps + kDeltaWarps - 1) / kDeltaWarps;
      if (blocks > (int64_t)st->sms * 16) blocks = (int64_t)st->sms * 16;
      const int ts = trace_pre(s);
      const cudaError_t e = launch_kernel(k_attn_delta, dim3((unsigned)blocks), dim3(kDeltaWarps * 32), 0, s, 1, 1,
                                          (const uint16_t*)dO, (const uint16_t*)O, delta, tokens, h, nh, L);
      trace_post(ts, s, kTraceSoftmax, tokens, h, 0);
      rc = launch_check(e, "softmax-gradient row sums");
      if (rc) return rc;
    }
    rc = attn_core_bwd_fused(st, QKV, P, dO, delta, dS, dQKV, h, nh, L, ns, s);
    if (rc) return rc;
    rc = gemm_batched(st, {dS, false, L, L, L, LL, nh * LL}, {QKV + h, true, d, L, h3, d, L * h3},
                      {dQKV, d, L, h3, d, L * h3}, L, d, L, nh, ns, est, s, kTraceAttnGemm, kCausalKUpTo);
    if (rc) return rc;
  } else {
  // per (sequence, head): dV = P^T dO, dS = P (dO V^T - delta) / sqrt(d) with delta = rowsum(dO * O)
  // (fused: the product dO V^T never leaves the GEMM), dQ = dS K, dK = dS^T Q
  rc = gemm_batched(st, {P, true, L, L, L, LL, nh * LL}, {dO, true, d, L, h, d, (int64_t)L * h},
                    {dQKV + 2 * h, d, L, h3, d, L * h3}, L, d, L, nh, ns, est, s, kTraceAttnGemm, kCausalKFrom);
  if (rc) return rc;
  float* delta = dP;  // ns * nh * L floats of the fp32 workspace
  {
    const int64_t warps = tokens * nh;
    int64_t blocks = (warps + kDeltaWarps - 1) / kDeltaWarps;
    if (blocks > (int64_t)st->sms * 16) blocks = (int64_t)st->sms * 16;
    const int ts = trace_pre(s);
    const cudaError_t e = launch_kernel(k_attn_delta, dim3((unsigned)blocks), dim3(kDeltaWarps * 32), 0, s, 1, 1,
                                        (const uint16_t*)dO, (const uint16_t*)O, delta, tokens, h, nh, L);
    trace_post(ts, s, kTraceSoftmax, tokens, h, 0);
    rc = launch_check(e, "softmax-gradient row sums");
    if (rc) return rc;
  }
  EpiParams eg{};
  eg.kind = kEpiSoftmaxGrad;
  eg.in0 = P;
  eg.g_in = delta;
  eg.ld = L;
  eg.alpha = 1.0f / std::sqrt((float)d);
  rc = gemm_batched(st, {dO, false, L, d, h, d, (int64_t)L * h}, {QKV + 2 * h, false, L, d, h3, d, L * h3},
                    {dS, L, L, L, LL, nh * LL}, L, L, d, nh, ns, eg, s, kTraceAttnGemm, kCausalSkipUpper);
  if (rc) return rc;
  rc = gemm_batched(st, {dS, false, L, L, L, LL, nh * LL}, {QKV + h, true, d, L, h3, d, L * h3},
                    {dQKV, d, L, h3, d, L * h3}, L, d, L, nh, ns, est, s, kTraceAttnGemm, kCausalKUpTo);
  if (rc) return rc;
  rc = gemm_batched(st, {dS, true, L, L, L, LL, nh * LL}, {QKV, true, d, L, h3, d, L * h3},
                    {dQKV + h, d, L, h3, d, L * h3}, L, d, L, nh, ns, est, s, kTraceAttnGemm, kCausalKFrom);
  if (rc) return rc;
  }
  // dbqkv (+)= sum dQKV; dWqkv (+)= X^T dQKV; dX = [dOut +] dQKV Wqkv^T
  {
    const int ts = trace_pre(s);
    const cudaError_t e =
        launch_kernel(k_colsum_bf16, dim3((unsigned)((h3 + kColsPerCta - 1) / kColsPerCta), colsum_split(st, h3, k_colsum_bf16)),
                      dim3(kColThreads), 0, s, 1, colsum_split(st, h3, k_colsum_bf16), (const uint16_t*)dQKV, (int64_t)h3, dbqkv,
                      tokens,
                      (int)h3, acc);
    trace_post(ts, s, kTraceColsum, tokens, h3, 0);
    rc = launch_check(e, "bias-gradient column sum");
    if (rc) return rc;
  }
  // dWqkv reads a transposed copy X^T (K-major) when large enough, in the dS
  // workspace again: every product that reads dS precedes it on the stream
  EpiParams eq{};
  eq.kind = acc ? kEpiF32Add : kEpiF32Store;
  eq.ld = h3;
  eq.g_out = dWqkv;
  if (ds_holds_copy && wgrad_transposed(h, (int)h3, tokens, dS)) {
    rc = launch_transposes(s, tokens, h, TransposeJob{X, dS}, TransposeJob{nullptr, nullptr}, "transposed copy of X");
    if (rc) return rc;
    rc = gemm(st, dS, false, T, dQKV, true, h3, h, (int)h3, T, eq, s, kTraceAttnGemm);
  } else {
    rc = gemm(st, X, true, h, dQKV, true, h3, h, (int)h3, T, eq, s, kTraceAttnGemm);
  }
  if (rc) return rc;
  EpiParams ex{};
  ex.kind = kEpiResAdd;
  ex.ld = h;
  ex.in0 = residual_grad ? dOut : nullptr;
  ex.out0 = dX;
  return gemm(st, dQKV, false, h3, Wqkv, false, h3, T, h, (int)h3, ex, s, kTraceAttnGemm);
}

int mlp_sync_status(void* stream) {
  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc) return rc;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(MLP_ECUDA, "stream synchronize: %s", cudaGetErrorString(e));
  int word[2] = {0, 0};
  e = cudaMemcpy(word, st->status, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(MLP_ECUDA, "status read: %s", cudaGetErrorString(e));
  if (word[0] != 0) {
    const int zero[2] = {0, 0};
    cudaMemcpy(st->status, zero, sizeof(zero), cudaMemcpyHostToDevice);
    // a launch that gave up may have left split-tail or tile counters behind
    cudaMemset(st->split_flags, 0, sizeof(int) * kSplitSlots * kSplitRegions);
    cudaMemset(st->sched_ctr, 0, sizeof(int) * 2 * kSplitRegions);
    return fail(word[0], "a kernel gave up on a bounded wait (site %d)", word[1]);
  }
  return MLP_OK;
}

const char* mlp_last_error(void) { return g_last_error.c_str(); }

int mlp_dropout_mask(int h, int64_t tokens, float p, uint64_t seed, uint64_t token_offset, uint8_t* m,
                     void* stream) {
  if (h <= 0 || tokens <= 0 || tokens >= (int64_t)1 << 31 || !(p >= 0.0f && p < 1.0f))
    return fail(MLP_EINVAL, "mlp_dropout_mask: bad h, tokens or p");
  if (m == nullptr) return fail(MLP_EINVAL, "mlp_dropout_mask: m is NULL");
  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc) return rc;
  const DropoutParams drop = make_dropout(p, seed, token_offset, h);
  const cudaError_t e = launch_kernel(k_dropout_mask, dim3(st->sms * 4), dim3(256), 0,
                                      static_cast<cudaStream_t>(stream), 1, 1, m, tokens, h, drop);
  return launch_check(e, "dropout mask");
}

int mlp_gelu_probe(const float* x, int64_t n, float* y, float* dy, void* stream) {
  if (n <= 0 || x == nullptr || y == nullptr || dy == nullptr) return fail(MLP_EINVAL, "mlp_gelu_probe: bad arguments");
  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc) return rc;
  const cudaError_t e =
      launch_kernel(k_gelu_probe, dim3(st->sms * 4), dim3(256), 0, static_cast<cudaStream_t>(stream), 1, 1, x, n, y, dy);
  return launch_check(e, "gelu probe");
}

int mlp_wait_timeout_probe(uint64_t limit_ns, void* stream) {
  if (limit_ns > 1000000000ull) return fail(MLP_EINVAL, "mlp_wait_timeout_probe: limit above one second");
  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc) return rc;
  const cudaError_t e = launch_kernel(k_wait_timeout_probe, dim3(1), dim3(32), 0, static_cast<cudaStream_t>(stream),
                                      1, 1, st->status, limit_ns);
  return launch_check(e, "wait-timeout probe");
}

uint64_t mlp_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int mlp_set_cta_pair(int mode) {
  if (mode < -1 || mode > 1) return fail(MLP_EINVAL, "mlp_set_cta_pair: mode %d not in {-1, 0, 1}", mode);
  g_pair_mode.store(mode, std::memory_order_relaxed);
  return MLP_OK;
}

int mlp_set_dependent_launch(int enable) {
  if (enable != 0 && enable != 1) return fail(MLP_EINVAL, "mlp_set_dependent_launch: %d not in {0, 1}", enable);
  g_pdl.store(enable, std::memory_order_relaxed);
  return MLP_OK;
}

int mlp_set_attn_fused(int enable) {
  if (enable != 0 && enable != 1) return fail(MLP_EINVAL, "mlp_set_attn_fused: %d not in {0, 1}", enable);
  g_attn_fused.store(enable, std::memory_order_relaxed);
  return MLP_OK;
}

int mlp_set_tile_scheduler(int mode) {
  if (mode < -1 || mode > 1) return fail(MLP_EINVAL, "mlp_set_tile_scheduler: %d not in {-1, 0, 1}", mode);
  g_tile_sched.store(mode, std::memory_order_relaxed);
  return MLP_OK;
}

int mlp_set_wgrad_transpose(int mode) {
  if (mode < -1 || mode > 1) return fail(MLP_EINVAL, "mlp_set_wgrad_transpose: %d not in {-1, 0, 1}", mode);
  g_wgrad_transpose.store(mode, std::memory_order_relaxed);
  return MLP_OK;
}

int mlp_set_split_tail(int enable) {
  if (enable != 0 && enable != 1) return fail(MLP_EINVAL, "mlp_set_split_tail: %d not in {0, 1}", enable);
  g_split_tail.store(enable, std::memory_order_relaxed);
  return MLP_OK;
}

int mlp_trace_begin(int capacity) {
  if (capacity <= 0 || capacity > (1 << 20)) return fail(MLP_EINVAL, "mlp_trace_begin: capacity %d out of range", capacity);
  std::lock_guard<std::mutex> lock(g_trace_mu);
  if (g_trace.on) return fail(MLP_EINVAL, "mlp_trace_begin: a trace is already running");
  g_trace.ev = new cudaEvent_t[2 * (size_t)capacity];
  g_trace.entries = new TraceEntry[capacity];
  for (int i = 0; i < 2 * capacity; ++i) {
    cudaError_t e = cudaEventCreate(&g_trace.ev[i]);
    if (e != cudaSuccess) {
      for (int j = 0; j < i; ++j) cudaEventDestroy(g_trace.ev[j]);
      delete[] g_trace.ev;
      delete[] g_trace.entries;
      g_trace.ev = nullptr;
      g_trace.entries = nullptr;
      return fail(MLP_ECUDA, "mlp_trace_begin: cudaEventCreate: %s", cudaGetErrorString(e));
    }
  }
  g_trace.capacity = capacity;
  g_trace.count = 0;
  g_trace.on = true;
  return MLP_OK;
}

int mlp_trace_end(int max_entries, int* kinds, int64_t* mnk, float* ms) {
  std::lock_guard<std::mutex> lock(g_trace_mu);
  if (!g_trace.on) return fail(MLP_EINVAL, "mlp_trace_end: no trace is running");
  g_trace.on = false;
  const int n = g_trace.count < max_entries ? g_trace.count : max_entries;
  int rc = n;
  for (int i = 0; i < n; ++i) {
    cudaError_t e = cudaEventSynchronize(g_trace.ev[2 * i + 1]);
    float t = 0.0f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&t, g_trace.ev[2 * i], g_trace.ev[2 * i + 1]);
    if (e != cudaSuccess) {
      rc = fail(MLP_ECUDA, "mlp_trace_end: %s", cudaGetErrorString(e));
      break;
    }
    if (kinds) kinds[i] = g_trace.entries[i].kind;
    if (mnk) {
      mnk[3 * i] = g_trace.entries[i].m;
      mnk[3 * i + 1] = g_trace.entries[i].n;
      mnk[3 * i + 2] = g_trace.entries[i].k;
    }
    if (ms) ms[i] = t;
  }
  for (int i = 0; i < 2 * g_trace.capacity; ++i) cudaEventDestroy(g_trace.ev[i]);
  delete[] g_trace.ev;
  delete[] g_trace.entries;
  g_trace.ev = nullptr;
  g_trace.entries = nullptr;
  g_trace.capacity = 0;
  g_trace.count = 0;
  return rc;
}

}  // extern "C"
