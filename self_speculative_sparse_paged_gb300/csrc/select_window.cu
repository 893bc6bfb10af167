// Query-agnostic selection: the first num_sink positions of the prefix and the
// last `window` ones, for every (sequence, KV head).
//
// "Vegas: Self-Speculative Decoding with Verification-Guided Sparse
// Attention", gist.science technical summary, §1 "Problem": simple
// query-agnostic methods such as a sliding window select cheaply but draft
// poorly; Vegas replaces them with selection guided by the verify pass.  This
// kernel produces that baseline's index set in the same layout as the top-k
// select, so the same draft kernel consumes either.  Sink positions (the
// first tokens, kept by streaming-attention selectors) are optional.
//
//   T_b = [0, min(s, L_b)) U [max(s, L_b - w), L_b),  k_b = min(L_b, s + w),
// written ascending to out_idx[(b * Hkv + g) * k_max + j], j < k_b, -1 after.
#include "kernels.h"
#include "vegas_common.cuh"

namespace vegas {

__global__ void __launch_bounds__(256) select_window_kernel(const WindowParams p) {
  griddep_begin();
  const int g = blockIdx.x, b = blockIdx.y;
  int L = p.ctx_lens[b];
  if (L < 0) {
    if (threadIdx.x == 0 && g == 0) set_error(p.err, kErrDeviceFault);
    L = 0;
  }
  const int s = min(p.num_sink, L);
  const int k = min(L, p.num_sink + p.window);
  const int wbeg = max(p.num_sink, L - p.window);   // first window position
  if (g == 0 && threadIdx.x == 0) p.k_out[b] = k;
  int32_t* out = p.out_idx + (size_t(b) * p.hkv + g) * p.k_max;
  for (int j = threadIdx.x; j < p.k_max; j += blockDim.x)
    out[j] = j < k ? (j < s ? j : wbeg + (j - s)) : -1;
}

cudaError_t launch_select_window(const WindowParams& p, int batch, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.hkv, batch, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, select_window_kernel, p);
}

}  // namespace vegas
