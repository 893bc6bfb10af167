// Top-k selection of the captured scores, per (sequence, KV head).
//
// "Vegas: Self-Speculative Decoding with Verification-Guided Sparse
// Attention", gist.science technical summary, §2.A: the selected set is the
// argmax over |T| = k of the summed attention logits; the objective is a sum
// of per-position scores, so T is the k largest scores (ties to the lower
// position under this library's reading), returned ascending.
//
// Scores become order-preserving uint32 keys (larger float -> larger key,
// -0.0 equal to +0.0, NaN lowest).  One thread-block cluster per (KV head,
// sequence); each CTA keeps its chunk of keys in shared memory.  The k-th
// largest key tau is found by narrowing a key interval [klo, khi] that holds
// it, one 2048-bin histogram per level, summed over the cluster through
// distributed shared memory:
//   level 0 counts the values in 2048 equal bins of the unit's [min, max] (a
//           monotone map, so every bin is a key interval and the bins fill
//           evenly);
//   level 1 splits the chosen bin into 2048 equal sub-bins the same way;
//   later levels bin the keys in [klo, khi] by the 11 bits of key - klo just
//           below the span's top bit.
// From level 1 on, every bin also records its smallest and largest key, so
// the chosen bin gives the next [klo, khi] exactly and the search ends as soon
// as that interval holds one key value (usually after level 1; at most five
// levels).  Then every
// key > tau is taken and keys == tau in position order until k are chosen;
// warp ballots plus the warps' and CTAs' counts place each chosen position at
// its rank, so the output is ascending and deterministic.
#include <cooperative_groups.h>

#include "kernels.h"
#include "vegas_common.cuh"

namespace cg = cooperative_groups;

namespace vegas {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelMaxChunk = 32768;                 // keys per CTA
constexpr int kSelChunkQuantum = 8 * kSelThreads;   // chunks hold 8 keys per thread at a time
constexpr int kBins = 2048;                         // 4 per thread
constexpr int kLevelWords = 6 * kBins;              // two sets of {count, min key, max key}

// Larger float -> larger key; -0.0 equals +0.0; NaN below every number.
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) return 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Inverse of order_key on non-NaN keys.
__device__ __forceinline__ float key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

constexpr int kMaxSelCluster = 8;

// Binning of a level: value bins of [min, max] (counts only), sub-bins of the
// chosen value bin, bits of key - klo; kDone once [klo, khi] holds one key.
enum { kValueBins, kSubBins, kKeyBits, kDone };

constexpr uint32_t kKeyNegInf = 0x007fffffu;   // order_key(-inf)
constexpr uint32_t kKeyPosInf = 0xff800000u;   // order_key(+inf)

__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
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
    const uint32_t w = lane < kSelWarps ? warp_tot[lane] : 0u;
    uint32_t wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    warp_tot[lane] = wi - w;
    if (lane == 31) warp_tot[32] = wi;
  }
  __syncthreads();
  const uint32_t ex = warp_tot[warp] + inc - v;
  total = warp_tot[32];
  __syncthreads();
  return ex;
}

__global__ void __launch_bounds__(kSelThreads, 1) select_topk_kernel(const SelectParams p) {
  griddep_begin();
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int CL = (int)cluster.num_blocks();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = blockIdx.y, b = blockIdx.z;
  const int unit = b * p.hkv + g;

  extern __shared__ __align__(16) uint32_t smem[];
  uint32_t* cnt = smem;                    // [2][kBins] keys per bin (one set per level parity)
  uint32_t* bmn = smem + 2 * kBins;        // [2][kBins] smallest key of each bin
  uint32_t* bmx = smem + 4 * kBins;        // [2][kBins] largest key of each bin
  uint32_t* keys = smem + kLevelWords;     // [chunk]
  __shared__ uint32_t warp_tot[33];
  __shared__ uint32_t red[2 * kSelWarps];
  __shared__ uint32_t xch[4];              // read by the cluster: key range, then counts
  __shared__ uint32_t sel[4];              // chosen bin: keys above it, min and max key, index

  int L = p.ctx_lens[b];
  int k = p.k_per_seq[b];
  if (L < 0 || L > p.score_stride || k < 0 || k > L || k > p.k_max) {
    if (tid == 0 && rank == 0) set_error(p.err, kErrDeviceFault);
    L = max(0, min(L, p.score_stride));
    k = max(0, min(k, min(L, p.k_max)));
  }
  int32_t* out = p.out_idx + size_t(unit) * p.k_max;
  for (int j = k + rank * kSelThreads + tid; j < p.k_max; j += CL * kSelThreads) out[j] = -1;
  if (k == 0) return;   // uniform over the cluster
  if (k == L) {
    for (int j = rank * kSelThreads + tid; j < L; j += CL * kSelThreads) out[j] = j;
    return;
  }

  // Warp w owns chunk offsets r = 32 P w + 32 u + lane, u < P: contiguous per
  // warp, so position order is (rank, warp, u, lane).
  const int P = p.chunk / kSelThreads;
  const int start = rank * p.chunk;
  const int nvalid = max(0, min(p.chunk, L - start));
  const int r0 = warp * 32 * P + lane;
  const float* src = p.scores + size_t(unit) * p.score_stride + start;

  for (int i = tid; i < 2 * kBins; i += kSelThreads) {
    cnt[i] = 0u;
    bmn[i] = 0xffffffffu;
    bmx[i] = 0u;
  }
  uint32_t kmin = 0xffffffffu, kmax = 0u;
  for (int u0 = 0; u0 < P; u0 += 8) {
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = r0 + (u0 + i) * 32;
      v[i] = r < nvalid ? __ldcg(src + r) : 0.f;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = r0 + (u0 + i) * 32;
      if (r < nvalid) {
        const uint32_t key = order_key(v[i]);
        keys[r] = key;
        kmin = min(kmin, key);
        kmax = max(kmax, key);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  }
  if (lane == 0) {
    red[warp] = kmin;
    red[kSelWarps + warp] = kmax;
  }
  __syncthreads();
  if (tid == 0) {
    uint32_t a = 0xffffffffu, c = 0u;
    for (int w = 0; w < kSelWarps; ++w) {
      a = min(a, red[w]);
      c = max(c, red[kSelWarps + w]);
    }
    xch[0] = a;
    xch[1] = c;
  }
  cluster.sync();
  {
    uint32_t a[kMaxSelCluster], c[kMaxSelCluster];
#pragma unroll
    for (int q = 0; q < kMaxSelCluster; ++q) {
      if (q < CL) {
        const uint32_t* x = cluster.map_shared_rank(xch, q);
        a[q] = x[0];
        c[q] = x[1];
      }
    }
    kmin = 0xffffffffu;
    kmax = 0u;
#pragma unroll
    for (int q = 0; q < kMaxSelCluster; ++q) {
      if (q < CL) {
        kmin = min(kmin, a[q]);
        kmax = max(kmax, c[q]);
      }
    }
  }

  // ---- narrow [klo, khi] around the k-th largest key
  uint32_t need = (uint32_t)k;    // keys still to take inside [klo, khi]
  uint32_t klo = kmin, khi = kmax;
  const float vmin = key_value(kmin), vmax = key_value(kmax);
  const float range = vmax - vmin;
  // Value bins only over a finite, nonzero range.  t = (value - vmin) * scale
  // is evaluated identically (no contraction) wherever it is used.
  const bool linear = kmin > kKeyNegInf && kmax < kKeyPosInf && range > 1.0e-30f && range < 3.0e38f;
  const float scale = linear ? float(kBins) / range : 0.f;
  int mode = klo == khi ? kDone : (linear ? kValueBins : kKeyBits);
  uint32_t vbin = 0;              // chosen value bin (kSubBins)
  for (int level = 0; mode != kDone; ++level) {
    const int s = (level & 1) * kBins;
    const int lo = mode == kKeyBits ? max(0, (32 - __clz(khi - klo)) - 11) : 0;
    for (int u = 0; u < P; ++u) {
      const int r = r0 + u * 32;
      if (r >= nvalid) break;
      const uint32_t key = keys[r];
      uint32_t d;
      if (mode == kKeyBits) {
        if (key < klo || key > khi) continue;
        d = (key - klo) >> lo;
      } else {
        const float t = __fmul_rn(__fsub_rn(key_value(key), vmin), scale);
        const uint32_t bin = min((uint32_t)kBins - 1u, __float2uint_rz(fmaxf(0.f, t)));
        if (mode == kValueBins) {       // counts only: every key takes part
          atomicAdd(&cnt[s + bin], 1u);
          continue;
        }
        if (bin != vbin) continue;
        // t - vbin is exact (Sterbenz) and the scaling by 2048 too: monotone in the key
        d = min((uint32_t)kBins - 1u,
                __float2uint_rz(fmaxf(0.f, __fmul_rn(__fsub_rn(t, float(vbin)), float(kBins)))));
      }
      atomicAdd(&cnt[s + d], 1u);
      atomicMin(&bmn[s + d], key);
      atomicMax(&bmx[s + d], key);
    }
    cluster.sync();
    // The other set's last readers (the previous level) are past this barrier.
    for (int i = tid; i < kBins; i += kSelThreads) {
      cnt[(kBins - s) + i] = 0u;
      bmn[(kBins - s) + i] = 0xffffffffu;
      bmx[(kBins - s) + i] = 0u;
    }
    // Thread t owns bins b0 + 3 .. b0 (descending), b0 = kBins - 4 (t + 1).
    const int b0 = kBins - 4 * (tid + 1);
    uint4 x[kMaxSelCluster];
#pragma unroll
    for (int q = 0; q < kMaxSelCluster; ++q)
      if (q < CL) x[q] = *reinterpret_cast<const uint4*>(cluster.map_shared_rank(cnt + s + b0, q));
    uint32_t h3 = 0, h2 = 0, h1 = 0, h0 = 0;
#pragma unroll
    for (int q = 0; q < kMaxSelCluster; ++q) {
      if (q < CL) {
        h3 += x[q].w;
        h2 += x[q].z;
        h1 += x[q].y;
        h0 += x[q].x;
      }
    }
    uint32_t total;
    uint32_t above = block_exclusive_scan(h3 + h2 + h1 + h0, warp_tot, total);
    int chosen = -1;
    if (above < need && need <= above + h3) chosen = b0 + 3;
    else if ((above += h3) < need && need <= above + h2) chosen = b0 + 2;
    else if ((above += h2) < need && need <= above + h1) chosen = b0 + 1;
    else if ((above += h1) < need && need <= above + h0) chosen = b0;
    if (chosen >= 0) {
      uint32_t a = 0xffffffffu, c = 0u;
      if (mode != kValueBins) {
        uint32_t mn[kMaxSelCluster], mx[kMaxSelCluster];
#pragma unroll
        for (int q = 0; q < kMaxSelCluster; ++q) {
          if (q < CL) {
            mn[q] = cluster.map_shared_rank(bmn + s, q)[chosen];
            mx[q] = cluster.map_shared_rank(bmx + s, q)[chosen];
          }
        }
#pragma unroll
        for (int q = 0; q < kMaxSelCluster; ++q) {
          if (q < CL) {
            a = min(a, mn[q]);
            c = max(c, mx[q]);
          }
        }
      }
      sel[0] = above;
      sel[1] = a;
      sel[2] = c;
      sel[3] = (uint32_t)chosen;
    }
    __syncthreads();
    need -= sel[0];
    if (mode == kValueBins) {
      vbin = sel[3];
      mode = kSubBins;
    } else {
      klo = sel[1];
      khi = sel[2];
      mode = klo == khi ? kDone : kKeyBits;
    }
    __syncthreads();   // sel is rewritten by the next level
  }
  const uint32_t tau = klo;       // `need` keys equal to tau are taken, lowest positions first

  // ---- compaction in position order
  uint32_t n_gt = 0, n_eq = 0;
  for (int u = 0; u < P; ++u) {
    const int r = r0 + u * 32;
    const bool valid = r < nvalid;
    const uint32_t key = valid ? keys[r] : 0u;
    n_gt += __popc(__ballot_sync(0xffffffffu, valid && key > tau));
    n_eq += __popc(__ballot_sync(0xffffffffu, valid && key == tau));
  }
  if (lane == 0) {
    red[warp] = n_gt;
    red[kSelWarps + warp] = n_eq;
  }
  __syncthreads();
  if (warp == 0) {
    const uint32_t a = lane < kSelWarps ? red[lane] : 0u;
    const uint32_t c = lane < kSelWarps ? red[kSelWarps + lane] : 0u;
    uint32_t ia = a, ic = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t ta = __shfl_up_sync(0xffffffffu, ia, o);
      const uint32_t tc = __shfl_up_sync(0xffffffffu, ic, o);
      if (lane >= o) {
        ia += ta;
        ic += tc;
      }
    }
    if (lane < kSelWarps) {
      red[lane] = ia - a;
      red[kSelWarps + lane] = ic - c;
    }
    if (lane == 31) {
      xch[2] = ia;
      xch[3] = ic;
    }
  }
  cluster.sync();
  uint32_t gt = red[warp], eq = red[kSelWarps + warp];   // selected keys before this warp's
  {
    uint32_t a[kMaxSelCluster - 1], c[kMaxSelCluster - 1];
#pragma unroll
    for (int q = 0; q < kMaxSelCluster - 1; ++q) {
      if (q < rank) {
        const uint32_t* x = cluster.map_shared_rank(xch, q);
        a[q] = x[2];
        c[q] = x[3];
      }
    }
#pragma unroll
    for (int q = 0; q < kMaxSelCluster - 1; ++q) {
      if (q < rank) {
        gt += a[q];
        eq += c[q];
      }
    }
  }
  cluster_arrive();   // this CTA reads no other CTA's shared memory after here
  const uint32_t below = (1u << lane) - 1u;
  for (int u = 0; u < P; ++u) {
    const int r = r0 + u * 32;
    const bool valid = r < nvalid;
    const uint32_t key = valid ? keys[r] : 0u;
    const bool is_gt = valid && key > tau, is_eq = valid && key == tau;
    const uint32_t bg = __ballot_sync(0xffffffffu, is_gt);
    const uint32_t be = __ballot_sync(0xffffffffu, is_eq);
    const uint32_t gt_before = gt + __popc(bg & below);
    const uint32_t eq_before = eq + __popc(be & below);
    if (is_gt) out[gt_before + min(eq_before, need)] = start + r;
    else if (is_eq && eq_before < need) out[gt_before + eq_before] = start + r;
    gt += __popc(bg);
    eq += __popc(be);
  }
  cluster_wait();     // no CTA leaves while another may still read its shared memory
}

size_t select_smem_bytes(int chunk) { return size_t(kLevelWords + chunk) * 4; }

cudaError_t launch_select(const SelectParams& p, int cluster, int batch, cudaStream_t stream) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(select_topk_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)select_smem_bytes(kSelMaxChunk));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster, p.hkv, batch);
  cfg.blockDim = dim3(kSelThreads, 1, 1);
  cfg.dynamicSmemBytes = select_smem_bytes(p.chunk);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, select_topk_kernel, p);
}

int select_max_chunk() { return kSelMaxChunk; }
int select_chunk_quantum() { return kSelChunkQuantum; }

}  // namespace vegas
