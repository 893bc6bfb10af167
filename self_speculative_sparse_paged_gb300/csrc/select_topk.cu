// Top-k selection of the captured scores, per (sequence, KV head).
//
// "Vegas: Self-Speculative Decoding with Verification-Guided Sparse
// Attention", gist.science technical summary, §2.A: the selected set is the
// argmax over |T| = k of the summed attention logits; the objective is a sum
// of per-position scores, so T is the k largest scores (ties to the lower
// position under this library's reading), returned ascending.
//
// One thread-block cluster of CL CTAs per (KV head, sequence); CTA r keeps
// keys [r * chunk, (r + 1) * chunk) in shared memory as order-preserving
// uint32 keys.  Four radix passes of 8 bits find the k-th largest key tau:
// every CTA histograms the keys that match the prefix found so far, the
// cluster barrier publishes the histograms, and every CTA sums all CL of them
// through distributed shared memory and scans the 256 digits from the top.
// Then keys > tau are all taken and keys == tau are taken in position order
// until k are chosen; a per-thread contiguous segment, block scans and the
// CTAs' counts exchanged over the cluster place every chosen position at its
// rank, so the output is ascending and deterministic.
#include <cooperative_groups.h>

#include "kernels.h"
#include "vegas_common.cuh"

namespace cg = cooperative_groups;

namespace vegas {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelMaxChunk = 32768;

// Larger float -> larger key; -0.0 equals +0.0; NaN below every number.
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) return 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive scan over the block; returns the exclusive prefix, sets total.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* warp_tot,
                                                         uint32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < kSelWarps ? warp_tot[lane] : 0u;
    uint32_t wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    if (lane < kSelWarps) warp_tot[lane] = wi - w;   // exclusive warp offsets
    if (lane == kSelWarps - 1) warp_tot[kSelWarps] = wi;
  }
  __syncthreads();
  const uint32_t ex = warp_tot[warp] + inc - v;
  total = warp_tot[kSelWarps];
  __syncthreads();
  return ex;
}

__global__ void __launch_bounds__(kSelThreads) select_topk_kernel(const SelectParams p) {
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int CL = (int)cluster.num_blocks();
  const int tid = threadIdx.x;
  const int g = blockIdx.y, b = blockIdx.z;
  const int unit = b * p.hkv + g;

  extern __shared__ uint32_t keys[];
  __shared__ uint32_t hist[2][256];
  __shared__ uint32_t warp_tot[kSelWarps + 1];
  __shared__ uint32_t cnts[2];
  __shared__ int s_digit;
  __shared__ uint32_t s_above;

  int L = p.ctx_lens[b];
  int k = p.k_per_seq[b];
  if (L < 0 || L > p.score_stride || k < 0 || k > L || k > p.k_max) {
    if (tid == 0 && rank == 0) set_error(p.err, kErrDeviceFault);
    L = max(0, min(L, p.score_stride));
    k = max(0, min(k, min(L, p.k_max)));
  }
  int32_t* out = p.out_idx + size_t(unit) * p.k_max;
  for (int j = k + rank * kSelThreads + tid; j < p.k_max; j += CL * kSelThreads) out[j] = -1;
  if (k == 0) return;
  if (k == L) {
    for (int j = rank * kSelThreads + tid; j < L; j += CL * kSelThreads) out[j] = j;
    return;
  }

  const int start = rank * p.chunk;
  const int cnt = max(0, min(L - start, p.chunk));
  const float* src = p.scores + size_t(unit) * p.score_stride + start;
  // Loads are issued in batches of 8 per thread before any of them is used.
  for (int i0 = 0; i0 < cnt; i0 += 8 * kSelThreads) {
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * kSelThreads + tid;
      v[u] = i < cnt ? __ldcg(&src[i]) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * kSelThreads + tid;
      if (i < cnt) keys[i] = order_key(v[u]);
    }
  }

  uint32_t prefix = 0u, pmask = 0u;
  uint32_t krem = (uint32_t)k;
  const int lane = tid & 31;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    uint32_t* h = hist[pass & 1];
    if (tid < 256) h[tid] = 0u;
    __syncthreads();
    // Lanes holding the same digit add once per warp (match.any), which keeps
    // the heavily shared top digits from serialising on one bank.
    for (int i0 = 0; i0 < cnt; i0 += kSelThreads) {
      const int i = i0 + tid;
      const uint32_t key = i < cnt ? keys[i] : 0u;
      const bool in = i < cnt && (key & pmask) == prefix;
      const uint32_t digit = in ? ((key >> shift) & 255u) : 256u;
      const uint32_t peers = __match_any_sync(0xffffffffu, digit);
      if (in && lane == __ffs(peers) - 1) atomicAdd(&h[digit], (uint32_t)__popc(peers));
    }
    cluster.sync();
    uint32_t v = 0u;
    if (tid < 256) {
      for (int r = 0; r < CL; ++r) v += cluster.map_shared_rank(h, r)[255 - tid];
    }
    uint32_t tot;
    const uint32_t ex = block_exclusive_scan(v, warp_tot, tot);
    if (tid < 256 && ex < krem && krem <= ex + v) {
      s_digit = 255 - tid;
      s_above = ex;
    }
    __syncthreads();
    prefix |= uint32_t(s_digit) << shift;
    pmask |= 0xFFu << shift;
    krem -= s_above;
  }
  const uint32_t tau = prefix;   // the k-th largest key; krem keys equal to it are taken

  const int seg = (cnt + kSelThreads - 1) / kSelThreads;
  const int i0 = min(tid * seg, cnt), i1 = min(i0 + seg, cnt);
  uint32_t n_gt = 0u, n_eq = 0u;
  for (int i = i0; i < i1; ++i) {
    const uint32_t key = keys[i];
    n_gt += key > tau;
    n_eq += key == tau;
  }
  uint32_t gt_cta, eq_cta;
  const uint32_t gt_before = block_exclusive_scan(n_gt, warp_tot, gt_cta);
  const uint32_t eq_before = block_exclusive_scan(n_eq, warp_tot, eq_cta);
  if (tid == 0) {
    cnts[0] = gt_cta;
    cnts[1] = eq_cta;
  }
  cluster.sync();
  uint32_t gt_prev = 0u, eq_prev = 0u;
  for (int r = 0; r < rank; ++r) {
    const uint32_t* c = cluster.map_shared_rank(cnts, r);
    gt_prev += c[0];
    eq_prev += c[1];
  }
  const uint32_t quota = krem > eq_prev ? min(krem - eq_prev, eq_cta) : 0u;
  const uint32_t base = gt_prev + min(eq_prev, krem);
  uint32_t take_eq = quota > eq_before ? min(quota - eq_before, n_eq) : 0u;
  uint32_t pos = base + gt_before + min(eq_before, quota);
  for (int i = i0; i < i1; ++i) {
    const uint32_t key = keys[i];
    bool sel = key > tau;
    if (key == tau && take_eq > 0u) {
      sel = true;
      --take_eq;
    }
    if (sel) out[pos++] = start + i;
  }
  cluster.sync();   // no CTA leaves while another may still read its shared memory
}

cudaError_t launch_select(const SelectParams& p, int cluster, int batch, cudaStream_t stream) {
  const size_t smem = size_t(p.chunk) * 4;
  static size_t configured_smem = 0;
  static bool nonportable = false;
  if (smem > configured_smem) {
    cudaError_t e = cudaFuncSetAttribute(select_topk_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured_smem = smem;
  }
  if (cluster > 8 && !nonportable) {
    cudaError_t e = cudaFuncSetAttribute(select_topk_kernel,
                                         cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    nonportable = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster, p.hkv, batch);
  cfg.blockDim = dim3(kSelThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, select_topk_kernel, p);
}

int select_max_chunk() { return kSelMaxChunk; }

}  // namespace vegas
