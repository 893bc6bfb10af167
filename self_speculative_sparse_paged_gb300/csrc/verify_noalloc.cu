// Verify attention for callers that cannot allocate device memory.
//
// vegas_verify_attn_capture needs a caller-allocated workspace for its
// split-KV partial results.  Some callers have no way to provide one: a plugin
// whose host framework owns every device allocation through its own pool, or a
// latency-critical decode loop that must never call cudaMalloc (which can
// synchronise the whole device).  This entry point runs the same kernel with
// the workspace taken from a fixed array in this library's device memory.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds kScratchBytes of it until the process exits.  In host code its
// name is only a host-side stand-in, never a device address; the address the
// kernel gets comes from cudaGetSymbolAddress, fetched once per device (with
// that device current) on the first call there.  That first call on a device
// should therefore come before any stream capture.
//
// All calls share the one array: once a call's arguments have passed their
// checks, the kernel's per-unit counters are cleared on the stream just before
// the launch (a rejected call touches nothing), and calls whose work overlaps
// on the GPU (other streams, other host threads) race on the array.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/vegas.h"
#include "kernels.h"

#define VEGAS_API extern "C" __attribute__((visibility("default")))

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;   // 16 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_verify_scratch[kScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_dev[kMaxDevices] = {};

// Device address of g_verify_scratch on the current device (set-up on first use).
vegas_status_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return (vegas_status_t)vegas::record_failure(VEGAS_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return (vegas_status_t)vegas::record_failure(VEGAS_ERR_UNSUPPORTED, "device ordinal out of range");
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_dev[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_verify_scratch);
    if (e != cudaSuccess)
      return (vegas_status_t)vegas::record_failure(VEGAS_ERR_CUDA, cudaGetErrorString(e));
    g_scratch_dev[dev] = p;
  }
  *out = g_scratch_dev[dev];
  return VEGAS_OK;
}

// vegas::ScratchFn: the array on the current device, asked for only once the
// call's arguments have passed their checks.
vegas_status_t scratch_workspace(void** ws, size_t* bytes) {
  vegas_status_t st = scratch_address(ws);
  if (st == VEGAS_OK) *bytes = kScratchBytes;
  return st;
}

}  // namespace

VEGAS_API size_t vegas_verify_noalloc_max_scratch_bytes(void) { return kScratchBytes; }

VEGAS_API vegas_status_t vegas_verify_attn_capture_noalloc(
    const vegas_paged_kv_t* kv, const void* q, void* out, float* scores, int score_stride,
    const int32_t* ctx_lens, int batch, int gamma, int capture_row_a, int capture_row_b,
    float softmax_scale, void* stream) {
  // Every argument is checked before the array is touched; its counters are
  // then cleared on `stream` right before the kernel.
  vegas_status_t st = vegas::verify_two_rows(kv, q, out, scores, score_stride, ctx_lens, batch,
                                             gamma, capture_row_a, capture_row_b, softmax_scale,
                                             nullptr, 0, stream, scratch_workspace);
  if (st == VEGAS_ERR_WORKSPACE_TOO_SMALL)
    return (vegas_status_t)vegas::record_failure(
        st, "this shape needs more split-KV scratch than the fixed 16 MiB array; "
            "use vegas_verify_attn_capture with a caller-allocated workspace");
  return st;
}
