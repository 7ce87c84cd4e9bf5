// mlp_fwd_static_scratch: the forward of the MLP block for callers that cannot
// allocate device memory.
//
// One-slice forward calls (slice = i, t > 1) need an fp32 [tokens, h] workspace
// in which the row-split partial products Y_i B_i of successive calls are summed.
// mlp_fwd takes that workspace from the caller.  Some callers cannot provide one:
// a plugin that runs inside a host application owning all device memory through
// its own pool (the plugin has no allocator of its own and must not call
// cudaMalloc), or a latency-bound serving loop that may not allocate once it runs,
// because cudaMalloc/cudaFree can synchronise the device.  This entry point keeps
// the workspace in a fixed array in the library's own device memory instead.
//
// The array below is a file-scope __device__ variable: every GPU that loads the
// library holds it (16 MiB) until the process exits.  In host code its name is
// only a host-side stand-in, not a device address, so the device address is
// looked up once per device with cudaGetSymbolAddress while that device is
// current, and that address is what the kernels receive.
#include <cstdio>
#include <mutex>

#include <cuda_runtime.h>

#include "gb_mlp.h"

namespace gbmlp {
// Sets the message mlp_last_error() returns (defined with the other entry points).
void set_last_error(const char* msg);
}  // namespace gbmlp

namespace {

constexpr long long kScratchFloats = 4ll << 20;  // 16 MiB of fp32: tokens * h <= 4,194,304

static __device__ __align__(256) float g_fwd_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
float* g_scratch_dev[kMaxDevices] = {};

// The device address of the scratch array on the current device; looked up on
// the first call per device.  Returns MLP_OK or an error code.
int scratch_address(float** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return MLP_EUNSUPPORTED;
  if (dev < 0 || dev >= kMaxDevices) return MLP_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_dev[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_fwd_scratch);
    if (e != cudaSuccess || p == nullptr) {
      char msg[256];
      snprintf(msg, sizeof(msg), "mlp_fwd_static_scratch: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
      gbmlp::set_last_error(msg);
      return MLP_ECUDA;
    }
    g_scratch_dev[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_dev[dev];
  return MLP_OK;
}

}  // namespace

extern "C" int mlp_fwd_static_scratch(int h, int ffn, int t, int slice, int64_t tokens, float p, uint64_t seed,
                                      uint64_t token_offset, const mlp_bf16* X, const mlp_bf16* A, const mlp_bf16* a,
                                      const mlp_bf16* B, const mlp_bf16* b, const mlp_bf16* R, mlp_bf16* U,
                                      mlp_bf16* Y, mlp_bf16* O, void* stream) {
  // Other argument errors are reported by mlp_fwd, which checks everything else.
  if (h > 0 && tokens > 0 && (long long)tokens * (long long)h > kScratchFloats) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "mlp_fwd_static_scratch: tokens * h = %lld exceeds the built-in workspace of %lld floats",
             (long long)tokens * (long long)h, kScratchFloats);
    gbmlp::set_last_error(msg);
    return MLP_EINVAL;
  }
  float* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc == MLP_EUNSUPPORTED) {
    gbmlp::set_last_error("mlp_fwd_static_scratch: no CUDA device");
    return rc;
  }
  if (rc != MLP_OK) return rc;
  return mlp_fwd(h, ffn, t, slice, tokens, p, seed, token_offset, X, A, a, B, b, R, U, Y, scratch, O, stream);
}
