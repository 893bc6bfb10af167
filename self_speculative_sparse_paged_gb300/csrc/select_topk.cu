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
// it, one 2048-bin histogram per level:
//   level 0 counts the values in 2048 equal bins of the unit's [min, max] (a
//           monotone map, so every bin is a key interval and the bins fill
//           evenly);
//   level 1 splits the chosen bin into 2048 equal sub-bins the same way;
//   later levels bin the keys in [klo, khi] by the 11 bits of key - klo just
//           below the span's top bit.
// From level 1 on, every bin also records its smallest and largest key, so
// the chosen bin gives the next [klo, khi] exactly and the search ends as soon
// as that interval holds one key value (usually after level 1).  With more
// than eight keys a thread, a level-0 bin holding at most 256 keys over the
// cluster is resolved without level 1: every CTA sends its keys of the bin to
// every CTA, and each CTA ranks them locally.
//
// Each CTA also sums its histogram into 64 super-bins of 32 bins and pushes
// them (and, once, its key range) into every CTA of the cluster with remote
// stores.  After one cluster barrier per level, warp 0 of every CTA scans the
// super-bin counts locally and reads the counts and key bounds of the 32 bins
// of the chosen super-bin from every CTA through distributed shared memory:
// one small remote read per level instead of every CTA reading every
// histogram.  The same reads give, per CTA
// of the cluster, how many of its keys lie above the chosen bin (and, at the
// last level, inside it), so each CTA knows how many chosen positions precede
// its own without another exchange.  Every key > tau is taken and keys == tau
// in position order until k are chosen; warp ballots place each chosen
// position at its rank, so the output is ascending and deterministic.
//
// Shared mode (one T per sequence for every query head: the §2.A sum taken over
// all heads instead of each KV head's group): the keys are the fp32 sums of the
// sequence's KV-head score rows in head order, and the chosen positions are
// written to every KV head's row.
#include <cooperative_groups.h>

#include "kernels.h"
#include "vegas_common.cuh"

namespace cg = cooperative_groups;

namespace vegas {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelMaxChunk = 32768;                 // keys per CTA
constexpr int kSelChunkQuantum = 8 * kSelThreads;   // chunks are 1, 2, 4 or 8 quanta (8-64 keys a thread)
constexpr int kBins = 2048;
constexpr int kSuper = 64;                          // super-bins of kFine bins
constexpr int kFine = kBins / kSuper;               // 32: one per lane
constexpr int kMaxSelCluster = 8;
// two sets (one per level parity) of {count, min key, max key} per bin, and of
// every CTA's super-bin counts
constexpr int kLevelWords = 6 * kBins + 2 * kMaxSelCluster * kSuper;
// With more than eight keys a thread, a chosen value bin holding at most this
// many keys over the cluster is resolved from its keys directly instead of by
// a second histogram level.  (At eight keys a thread the extra code measured
// slower than the second level it saves.)
constexpr int kMaxCand = 256;
constexpr int kCandWords = kMaxCand + 4;   // the keys, then count, tau, keys above tau

// Binning of a level: value bins of [min, max] (counts only), sub-bins of the
// chosen value bin, bits of key - klo; kDone once [klo, khi] holds one key.
enum { kValueBins, kSubBins, kKeyBits, kDone };

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

constexpr uint32_t kKeyNegInf = 0x007fffffu;   // order_key(-inf)
constexpr uint32_t kKeyPosInf = 0xff800000u;   // order_key(+inf)

// First half of the exit barrier: this CTA reads no other CTA's shared memory
// from here on.  Every remote read before it has already been consumed, so
// the arrival publishes nothing and needs no release ordering.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t warp_sum(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ uint32_t warp_inclusive_scan(uint32_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// Shared state of the level search, written by warp 0.
struct SelState {
  uint32_t bin, above, klo, khi;
  uint32_t gt[kMaxSelCluster];    // per CTA: keys above the chosen bins so far
  uint32_t in[kMaxSelCluster];    // per CTA: keys inside this level's chosen bin
};

// Warp 0: finds the bin holding the need-th largest key from the cluster's
// histograms of one set (counts `cnt` and key bounds `bmn`/`bmx`, unless
// `bounds` is false, read remotely; super-bin counts of every CTA in the local
// `sup_all`) and records it in `st`.
__device__ __forceinline__ void search_level(cg::cluster_group& cluster, int CL,
                                             const uint32_t* cnt, const uint32_t* sup_all,
                                             const uint32_t* bmn, const uint32_t* bmx,
                                             bool bounds, uint32_t need, SelState& st) {
  const int lane = threadIdx.x & 31;
  // super-bins 63 - 2 lane (hi) and 62 - 2 lane (lo): descending with the lane;
  // every CTA's counts were pushed into this CTA's sup_all[q][kSuper]
  const int sbh = kSuper - 1 - 2 * lane, sbl = sbh - 1;
  uint32_t ch[kMaxSelCluster], cl[kMaxSelCluster];
#pragma unroll
  for (int q = 0; q < kMaxSelCluster; ++q) {
    ch[q] = cl[q] = 0u;
    if (q < CL) {
      const uint2 x = *reinterpret_cast<const uint2*>(sup_all + q * kSuper + sbl);
      cl[q] = x.x;
      ch[q] = x.y;
    }
  }
  uint32_t th = 0, tl = 0;
#pragma unroll
  for (int q = 0; q < kMaxSelCluster; ++q) {
    th += ch[q];
    tl += cl[q];
  }
  const uint32_t incl = warp_inclusive_scan(th + tl), excl = incl - th - tl;
  const bool hit = excl < need && need <= incl;
  const int hlane = __ffs(__ballot_sync(0xffffffffu, hit)) - 1;
  int sb = 0;
  uint32_t above = 0;
  if (hit) {
    if (need <= excl + th) {
      sb = sbh;
      above = excl;
    } else {
      sb = sbl;
      above = excl + th;
    }
  }
  sb = __shfl_sync(0xffffffffu, sb, hlane);
  above = __shfl_sync(0xffffffffu, above, hlane);
  // the 32 bins of super-bin sb, bin sb * 32 + 31 - lane (descending with the lane)
  const int fb = sb * kFine + (kFine - 1 - lane);
  // counts and key bounds of the lane's bin in every CTA, in one round trip
  uint32_t f[kMaxSelCluster], fmn[kMaxSelCluster], fmx[kMaxSelCluster];
#pragma unroll
  for (int q = 0; q < kMaxSelCluster; ++q) {
    f[q] = 0u;
    fmn[q] = 0xffffffffu;
    fmx[q] = 0u;
    if (q < CL) {
      f[q] = cluster.map_shared_rank(cnt, q)[fb];
      if (bounds) {
        fmn[q] = cluster.map_shared_rank(bmn, q)[fb];
        fmx[q] = cluster.map_shared_rank(bmx, q)[fb];
      }
    }
  }
  uint32_t ft = 0;
#pragma unroll
  for (int q = 0; q < kMaxSelCluster; ++q) ft += f[q];
  const uint32_t fincl = warp_inclusive_scan(ft), fexcl = fincl - ft;
  const uint32_t need2 = need - above;
  const bool hit2 = fexcl < need2 && need2 <= fincl;
  const int hl2 = __ffs(__ballot_sync(0xffffffffu, hit2)) - 1;
  const int bin = sb * kFine + (kFine - 1 - hl2);
  const uint32_t above_bin = above + __shfl_sync(0xffffffffu, fexcl, hl2);
  // per CTA: keys in bins above the chosen one (summed over the lanes by a
  // reduce-scatter: lane 4q ends with CTA q's sum), and inside it
  uint32_t up[kMaxSelCluster];
#pragma unroll
  for (int q = 0; q < kMaxSelCluster; ++q)
    up[q] = (sbh > sb ? ch[q] : 0u) + (sbl > sb ? cl[q] : 0u) + (lane < hl2 ? f[q] : 0u);
  static_assert(kMaxSelCluster == 8, "three halving rounds");
#pragma unroll
  for (int r = 0, w = kMaxSelCluster / 2; w >= 1; ++r, w >>= 1) {
    const bool hi = lane & (16 >> r);   // keeps the upper w of the 2w values held
#pragma unroll
    for (int j = 0; j < w; ++j) {
      const uint32_t send = hi ? up[j] : up[j + w];
      up[j] = (hi ? up[j + w] : up[j]) + __shfl_xor_sync(0xffffffffu, send, 16 >> r);
    }
  }
  up[0] += __shfl_xor_sync(0xffffffffu, up[0], 2);
  up[0] += __shfl_xor_sync(0xffffffffu, up[0], 1);
  uint32_t inq[kMaxSelCluster];
#pragma unroll
  for (int q = 0; q < kMaxSelCluster; ++q) inq[q] = __shfl_sync(0xffffffffu, f[q], hl2);
  if ((lane & 3) == 0 && (lane >> 2) < CL) st.gt[lane >> 2] += up[0];
  if (lane < CL) {
#pragma unroll
    for (int q = 0; q < kMaxSelCluster; ++q)
      if (q == lane) st.in[q] = inq[q];
  }
  // key bounds of the chosen bin over the cluster (held by lane hl2)
  uint32_t a = 0xffffffffu, z = 0u;
#pragma unroll
  for (int q = 0; q < kMaxSelCluster; ++q) {
    a = min(a, fmn[q]);
    z = max(z, fmx[q]);
  }
  a = __shfl_sync(0xffffffffu, a, hl2);
  z = __shfl_sync(0xffffffffu, z, hl2);
  if (lane == 0) {
    st.bin = (uint32_t)bin;
    st.above = above_bin;
    st.klo = a;
    st.khi = z;
  }
}

// P keys per thread (the CTA's chunk is kSelThreads * P keys); SHARED: one T per
// sequence from the sum over its KV heads.
template <int P, bool SHARED>
__global__ void __launch_bounds__(kSelThreads, 1) select_topk_kernel(const SelectParams p) {
  griddep_launch_dependents();
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int CL = (int)cluster.num_blocks();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = blockIdx.y, b = blockIdx.z;
  const int unit = b * p.hkv + g;

  extern __shared__ __align__(16) uint32_t smem[];
  uint32_t* cnt = smem;                    // [2][kBins] keys per bin
  uint32_t* bmn = smem + 2 * kBins;        // [2][kBins] smallest key of each bin
  uint32_t* bmx = smem + 4 * kBins;        // [2][kBins] largest key of each bin
  uint32_t* sup = smem + 6 * kBins;        // [2][kMaxSelCluster][kSuper] every CTA's super-bin counts
  uint32_t* keys = smem + kLevelWords;     // [chunk]
  // (P > 8) keys of the chosen value bin, by CTA; then count, tau, keys above tau
  uint32_t* cand = keys + p.chunk;
  __shared__ uint32_t red[2 * kSelWarps];
  __shared__ uint32_t xch[2 * kMaxSelCluster];   // every CTA's key range, pushed here
  __shared__ SelState st;
  // Both histogram sets are cleared before the wait for the previous kernel
  // (no global memory is touched before it).
  for (int i = tid; i < 2 * kBins; i += kSelThreads) {
    cnt[i] = 0u;
    bmn[i] = 0xffffffffu;
    bmx[i] = 0u;
  }
  if (tid < kMaxSelCluster) {
    st.gt[tid] = 0u;
    st.in[tid] = 0u;
  }
  if constexpr (P > 8) {
    if (tid < 4) cand[kMaxCand + tid] = 0u;
  }
  griddep_wait();

  // Warp w owns chunk offsets r = 32 P w + 32 u + lane, u < P: contiguous per
  // warp, so position order is (rank, warp, u, lane).  The first keys are
  // requested before the sequence length is known (within the score row).
  const int start = rank * p.chunk;
  const int lim = max(0, min(p.chunk, p.score_stride - start));
  const int r0 = warp * 32 * P + lane;
  const float* src = p.scores + size_t(unit) * p.score_stride + start;
  // one T per sequence: the fp32 sum of the sequence's KV-head rows, in head order
  const int nsum = SHARED ? p.hkv : 1;
  auto score_at = [&](int r) {
    float acc = __ldcg(src + r);
    for (int h = 1; h < nsum; ++h) acc += __ldcg(src + size_t(h) * p.score_stride + r);
    return acc;
  };
  float v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = r0 + i * 32;
    v[i] = r < lim ? score_at(r) : 0.f;
  }

  int L = p.ctx_lens[b];
  int k = p.k_per_seq[b];
  if (L < 0 || L > p.score_stride || k < 0 || k > L || k > p.k_max) {
    if (tid == 0 && rank == 0) set_error(p.err, kErrDeviceFault);
    L = max(0, min(L, p.score_stride));
    k = max(0, min(k, min(L, p.k_max)));
  }
  // output rows: this unit's, or (shared T) every KV head's row of the sequence
  int32_t* out = p.out_idx + size_t(unit) * p.k_max;
  const int nout = SHARED ? p.hkv : 1;
  auto put = [&](int j, int32_t v) {
    for (int h = 0; h < nout; ++h) out[size_t(h) * p.k_max + j] = v;
  };
  for (int j = k + rank * kSelThreads + tid; j < p.k_max; j += CL * kSelThreads) put(j, -1);
  if (k == 0) return;   // uniform over the cluster
  if (k == L) {
    for (int j = rank * kSelThreads + tid; j < L; j += CL * kSelThreads) put(j, j);
    return;
  }
  const int nvalid = max(0, min(p.chunk, L - start));

  // At eight keys a thread the keys stay in registers; larger chunks keep
  // them in shared memory.
  constexpr bool kRegKeys = P <= 8;
  uint32_t kreg[kRegKeys ? P : 1];
#pragma unroll
  for (int u = 0; u < (kRegKeys ? P : 1); ++u) kreg[u] = 0u;
  auto key_at = [&](int u, int r) {
    if constexpr (kRegKeys)
      return kreg[u];
    else
      return keys[r];
  };
  uint32_t kmin = 0xffffffffu, kmax = 0u;
#pragma unroll 1
  for (int u0 = 0; u0 < P; u0 += 8) {
    if (u0 > 0) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = r0 + (u0 + i) * 32;
        v[i] = r < nvalid ? score_at(r) : 0.f;
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = r0 + (u0 + i) * 32;
      if (r < nvalid) {
        const uint32_t key = order_key(v[i]);
        if constexpr (kRegKeys)
          kreg[u0 + i] = key;
        else
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
  if (warp == 0) {
    // this CTA's key range, pushed into every CTA of the cluster (lane q -> CTA q)
    uint32_t a = lane < kSelWarps ? red[lane] : 0xffffffffu;
    uint32_t c = lane < kSelWarps ? red[kSelWarps + lane] : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      a = min(a, __shfl_xor_sync(0xffffffffu, a, o));
      c = max(c, __shfl_xor_sync(0xffffffffu, c, o));
    }
    if (lane < CL) {
      uint32_t* x = cluster.map_shared_rank(xch, lane);
      x[2 * rank] = a;
      x[2 * rank + 1] = c;
    }
  }
  cluster.sync();
  kmin = 0xffffffffu;
  kmax = 0u;
  for (int q = 0; q < CL; ++q) {
    kmin = min(kmin, xch[2 * q]);
    kmax = max(kmax, xch[2 * q + 1]);
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
  const bool searched = mode != kDone;
  uint32_t vbin = 0;              // chosen value bin (kSubBins)
  for (int level = 0; mode != kDone; ++level) {
    const int s = level & 1;
    uint32_t* c = cnt + s * kBins;
    uint32_t* mn = bmn + s * kBins;
    uint32_t* mx = bmx + s * kBins;
    uint32_t* su = sup + s * kMaxSelCluster * kSuper;
    const int lo = mode == kKeyBits ? max(0, (32 - __clz(khi - klo)) - 11) : 0;
#pragma unroll 8
    for (int u = 0; u < P; ++u) {
      const int r = r0 + u * 32;
      if (r >= nvalid) continue;
      const uint32_t key = key_at(u, r);
      uint32_t d;
      if (mode == kKeyBits) {
        if (key < klo || key > khi) continue;
        d = (key - klo) >> lo;
      } else {
        const float t = __fmul_rn(__fsub_rn(key_value(key), vmin), scale);
        const uint32_t bin = min((uint32_t)kBins - 1u, __float2uint_rz(fmaxf(0.f, t)));
        if (mode == kValueBins) {       // counts only: every key takes part
          atomicAdd(&c[bin], 1u);
          continue;
        }
        if (bin != vbin) continue;
        // t - vbin is exact (Sterbenz) and the scaling by 2048 too: monotone in the key
        d = min((uint32_t)kBins - 1u,
                __float2uint_rz(fmaxf(0.f, __fmul_rn(__fsub_rn(t, float(vbin)), float(kBins)))));
      }
      atomicAdd(&c[d], 1u);
      atomicMin(&mn[d], key);
      atomicMax(&mx[d], key);
    }
    __syncthreads();
    // super-bin sums: thread t adds bins 4t .. 4t + 3, the eight threads of a
    // super-bin reduce with shuffles (each ends with the sum), and thread q of
    // the eight pushes it into CTA q's su[rank][.]: one remote store a thread
    // rather than one thread looping over the CTAs
    static_assert(4 * kSelThreads == kBins && kFine == 32, "four bins a thread");
    static_assert(kMaxSelCluster <= 8, "one CTA per thread of a super-bin");
    {
      const uint4 c4 = *reinterpret_cast<const uint4*>(c + 4 * tid);
      uint32_t x = c4.x + c4.y + c4.z + c4.w;
      x += __shfl_xor_sync(0xffffffffu, x, 1);
      x += __shfl_xor_sync(0xffffffffu, x, 2);
      x += __shfl_xor_sync(0xffffffffu, x, 4);
      if ((tid & 7) < CL) cluster.map_shared_rank(su, tid & 7)[rank * kSuper + (tid >> 3)] = x;
    }
    cluster.sync();
    // The other set's last readers (the previous level's search) are past
    // this barrier: clear it for the next level.
    {
      const int o = (s ^ 1) * kBins;
      for (int i = tid; i < kBins; i += kSelThreads) {
        cnt[o + i] = 0u;
        bmn[o + i] = 0xffffffffu;
        bmx[o + i] = 0u;
      }
    }
    if (warp == 0) search_level(cluster, CL, c, su, mn, mx, mode != kValueBins, need, st);
    __syncthreads();
    need -= st.above;
    if (mode == kValueBins) {
      vbin = st.bin;
      mode = kSubBins;
      uint32_t nb = 0, base = 0;   // keys in the chosen bin: all, and in the CTAs before this one
      for (int q = 0; q < CL; ++q) {
        nb += st.in[q];
        base += q < rank ? st.in[q] : 0u;
      }
      if (P > 8 && nb <= (uint32_t)kMaxCand) {
        uint32_t& ncand = cand[kMaxCand];
        uint32_t& cand_tau = cand[kMaxCand + 1];
        uint32_t& cand_above = cand[kMaxCand + 2];
        // Few keys in the chosen bin: every CTA pushes its keys of the bin
        // into every CTA's cand[] (CTA q's at the bin counts of the CTAs
        // before it), and each CTA finds tau, the need-th largest of them,
        // and the per-CTA counts above and at tau, locally.
#pragma unroll 8
        for (int u = 0; u < P; ++u) {
          const int r = r0 + u * 32;
          if (r >= nvalid) continue;
          const uint32_t key = key_at(u, r);
          const float t = __fmul_rn(__fsub_rn(key_value(key), vmin), scale);
          const uint32_t bin = min((uint32_t)kBins - 1u, __float2uint_rz(fmaxf(0.f, t)));
          if (bin != vbin) continue;
          const uint32_t j = base + atomicAdd(&ncand, 1u);
          if (j < (uint32_t)kMaxCand)   // always (the bin counts bound it)
            for (int q = 0; q < CL; ++q) cluster.map_shared_rank(cand, q)[j] = key;
        }
        cluster.sync();
        for (uint32_t t = tid; t < nb; t += kSelThreads) {
          const uint32_t kt = cand[t];
          uint32_t n_gt = 0, n_ge = 0;
          for (uint32_t j = 0; j < nb; ++j) {
            n_gt += cand[j] > kt ? 1u : 0u;
            n_ge += cand[j] >= kt ? 1u : 0u;
          }
          if (n_gt < need && need <= n_ge) {   // every such thread holds the same key
            cand_tau = kt;
            cand_above = n_gt;
          }
        }
        __syncthreads();
        const uint32_t tau_c = cand_tau;
        if (warp == 0) {
          // lane q < CL: CTA q's segment cand[b0, b0 + in[q])
          uint32_t b0 = 0, nq = 0;
          for (int q = 0; q < CL; ++q) {
            b0 += q < lane ? st.in[q] : 0u;
            nq = q == lane ? st.in[q] : nq;
          }
          __syncwarp();
          uint32_t a = 0, e = 0;
          for (uint32_t j = b0; j < b0 + nq; ++j) {
            a += cand[j] > tau_c ? 1u : 0u;
            e += cand[j] == tau_c ? 1u : 0u;
          }
          if (lane < CL) {
            st.gt[lane] += a;
            st.in[lane] = e;
          }
        }
        __syncthreads();
        need -= cand_above;
        klo = khi = tau_c;
        mode = kDone;
      }
    } else {
      klo = st.klo;
      khi = st.khi;
      mode = klo == khi ? kDone : kKeyBits;
    }
  }
  cluster_arrive();   // no shared memory of another CTA is read after this point
  const uint32_t tau = klo;       // `need` keys equal to tau are taken, lowest positions first

  // chosen keys before this CTA's (gt) and keys equal to tau before it (eq)
  uint32_t gt = 0, eq = 0;
  for (int q = 0; q < rank; ++q) {
    gt += searched ? st.gt[q] : 0u;
    eq += searched ? st.in[q] : (uint32_t)max(0, min(p.chunk, L - q * p.chunk));
  }

  // ---- compaction in position order: per-warp counts, then ballot ranks
  uint32_t n_gt = 0, n_eq = 0;
#pragma unroll 8
  for (int u = 0; u < P; ++u) {
    const int r = r0 + u * 32;
    const bool valid = r < nvalid;
    const uint32_t key = valid ? key_at(u, r) : 0u;
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
    const uint32_t ia = warp_inclusive_scan(a), ic = warp_inclusive_scan(c);
    __syncwarp();
    if (lane < kSelWarps) {
      red[lane] = ia - a;
      red[kSelWarps + lane] = ic - c;
    }
  }
  __syncthreads();
  gt += red[warp];
  eq += red[kSelWarps + warp];
  const uint32_t below = (1u << lane) - 1u;
#pragma unroll 8
  for (int u = 0; u < P; ++u) {
    const int r = r0 + u * 32;
    const bool valid = r < nvalid;
    const uint32_t key = valid ? key_at(u, r) : 0u;
    const bool is_gt = valid && key > tau, is_eq = valid && key == tau;
    const uint32_t bg = __ballot_sync(0xffffffffu, is_gt);
    const uint32_t be = __ballot_sync(0xffffffffu, is_eq);
    const uint32_t gt_before = gt + __popc(bg & below);
    const uint32_t eq_before = eq + __popc(be & below);
    if (is_gt) put(gt_before + min(eq_before, need), start + r);
    else if (is_eq && eq_before < need) put(gt_before + eq_before, start + r);
    gt += __popc(bg);
    eq += __popc(be);
  }
  cluster_wait();     // no CTA leaves while another may still read its shared memory
}

size_t select_smem_bytes(int chunk) {
  return size_t(kLevelWords + chunk + (chunk > 8 * kSelThreads ? kCandWords : 0)) * 4;
}

template <int P, bool SHARED>
static cudaError_t launch_select_p(const SelectParams& p, int cluster, int batch,
                                   cudaStream_t stream) {
  static std::atomic<uint32_t> configured{0};
  cudaError_t e = once_per_device(configured, [] {
    return cudaFuncSetAttribute(select_topk_kernel<P, SHARED>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)select_smem_bytes(P * kSelThreads));
  });
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster, p.shared ? 1 : p.hkv, batch);
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
  return cudaLaunchKernelEx(&cfg, select_topk_kernel<P, SHARED>, p);
}

template <bool SHARED>
static cudaError_t launch_select_s(const SelectParams& p, int cluster, int batch,
                                   cudaStream_t stream) {
  switch (p.chunk / kSelThreads) {
    case 8: return launch_select_p<8, SHARED>(p, cluster, batch, stream);
    case 16: return launch_select_p<16, SHARED>(p, cluster, batch, stream);
    case 32: return launch_select_p<32, SHARED>(p, cluster, batch, stream);
    case 64: return launch_select_p<64, SHARED>(p, cluster, batch, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_select(const SelectParams& p, int cluster, int batch, cudaStream_t stream) {
  return p.shared ? launch_select_s<true>(p, cluster, batch, stream)
                  : launch_select_s<false>(p, cluster, batch, stream);
}

int select_max_chunk() { return kSelMaxChunk; }
int select_chunk_quantum() { return kSelChunkQuantum; }

}  // namespace vegas
