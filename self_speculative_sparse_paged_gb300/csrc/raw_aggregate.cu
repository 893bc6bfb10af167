// The pages' capture, second half: per-(row, head) raw logits summed into one
// score per (position, KV head).
//
// "Vegas: Self-Speculative Decoding with Verification-Guided Sparse
// Attention", gist.science technical summary, §3 "Implementation": the verify
// kernel (FlashAttention-3 there) writes the raw pre-softmax logits of the
// collected rows to memory, and the selection objective of §2.A aggregates
// them over the rows and the query heads of each KV head afterwards.  This
// library fuses that sum into the verify kernel; this kernel and the raw mode
// of the verify kernels exist to measure the pages' way against it.
//
//   scores[(b * Hkv + g) * score_stride + i]
//     = sum_{r < R} sum_{hl < G} raw[((b * R + r) * Hq + g * G + hl) * raw_stride + i]
// for i < L_b, summed in fp32 in (r, hl) order.
#include "kernels.h"
#include "vegas_common.cuh"

namespace vegas {

__global__ void __launch_bounds__(256) raw_aggregate_kernel(const RawAggParams p) {
  griddep_begin();
  const int g = blockIdx.y, b = blockIdx.z;
  int L = p.ctx_lens[b];
  if (L < 0 || L > p.raw_stride || L > p.score_stride) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && g == 0) set_error(p.err, kErrDeviceFault);
    L = max(0, min(L, min(p.raw_stride, p.score_stride)));
  }
  const int G = p.hq / p.hkv;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < L; i += gridDim.x * blockDim.x) {
    float acc = 0.f;
    for (int r = 0; r < p.rows; ++r) {
      const float* src = p.raw + ((size_t(b) * p.rows + r) * p.hq + size_t(g) * G) * p.raw_stride + i;
      for (int hl = 0; hl < G; ++hl) acc += __ldcs(src + size_t(hl) * p.raw_stride);
    }
    p.scores[(size_t(b) * p.hkv + g) * p.score_stride + i] = acc;
  }
}

cudaError_t launch_raw_aggregate(const RawAggParams& p, int batch, int max_len,
                                 cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(max(1, min((max_len + 255) / 256, 64)), p.hkv, batch);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, raw_aggregate_kernel, p);
}

}  // namespace vegas
