// Verify attention with Collect-2-Query capture on the 5th-generation tensor
// cores (tcgen05, accumulators in tensor memory), head_dim 128 or 64 (this
// file is compiled once per head_dim, VEGAS_TC_D).
//
// Same contract as the mma.sync kernel in verify_attn.cu ("Vegas:
// Self-Speculative Decoding with Verification-Guided Sparse Attention",
// gist.science technical summary, §2 "Core mechanism", §2.A, §2.B
// "Collect-2-Query", §3 "Implementation"), used when the unit's query columns
// (the (gamma+1)*G rows plus the two capture columns) fit in 40 at head_dim
// 128 and 64 at head_dim 64.
//
// One CTA per (split, KV head, sequence), 12 warps:
//   warps 0, 10, 11  TMA producers (issue rate is per warp, so a tile's boxes
//              are spread over three warps): K and V tiles of 128 positions (8
//              pages) stream into K and V rings (3 + 3 slots; 3 + 4 at head_dim
//              64), block-table entries prefetched four tiles ahead;
//   warp 1     allocates tensor memory; the warp runs the MMA loop uniformly
//              and one elected lane issues
//                S^T[128 pos x N] = K[128 x D] . Q^T   (both K-major, the K
//                tile consumed straight from the TMA's 128-byte swizzle),
//                O^T[128 d x N]  += V^T[128 x 128] . P^T (V read MN-major; at
//                head_dim 64 the upper half of V^T is one shared region of
//                zeros with a ones row, so O^T row 64 sums P);
//   warps 2-5  softmax group 0 (even tiles), warps 6-9 group 1 (odd tiles):
//              thread i of a group owns tensor-memory lane i, i.e. tile
//              position i for S and head dimension i for its O^T accumulator.
// Each group keeps its own running maxima, row sums and O^T accumulator in
// tensor memory (the two are merged at the end, like two splits).  Per tile a
// softmax thread loads its position's logits, writes the captured score (the
// two capture columns hold the summed captured query, so the score is their
// sum), masks, and raises the running maxima only when a logit exceeds them by
// 8 (one vote per group); only then is the group's O^T rescaled in tensor
// memory.  It writes P^T = 2^(x - m) as bf16 (wide tiles: 2^y with y taken
// relative to a per-column reference in one FMA) into a 128-byte-swizzled
// shared buffer that the PV MMA reads (K-major up to 32 columns, MN-major for
// 64-column tiles).
//
// Splits of a unit merge either on chip, when all of them form one
// thread-block cluster (every group pushes its state to the rank that owns the
// output row, through distributed shared memory; no workspace), or through the
// workspace in the last-arriving CTA.
#include <cooperative_groups.h>

#include "kernels.h"

#ifndef VEGAS_TC_D
#error "compile with -DVEGAS_TC_D=64 or -DVEGAS_TC_D=128"
#endif
#include "split_merge.cuh"

namespace cg = cooperative_groups;

namespace vegas {

template <int D, int NQP, int NQC>
struct TcCfg {
  // K and V tiles live in separate rings: a K slot frees when its S MMA
  // completes, a V slot only when its PV MMA does.  Under full HBM load a
  // tile's load latency reaches ~2 us, which each ring must cover on its own.
  // (Two K slots when 64 query columns at head_dim 128 leave no room for three.)
  // (At head_dim 64 a V slot is half as large and the V ring is four deep: a
  // V slot is held from its load until its PV MMA has completed, so one more
  // slot keeps more of the stream in flight; five to seven slots, which let the
  // V loads run further ahead of the K loads, measured slower.)
  static constexpr int KS = (D == 128 && NQP == 64) ? 2 : 3;
  static constexpr int VS = D == 64 ? 4 : 3;
  static constexpr int kHalves = D / 64;             // 64-column (128-byte) halves of a row
  static constexpr int kKV = 128 * D * 2;            // one K tile (and one V tile)
  // The PV MMA's A operand (V^T) always spans 128 head dimensions: at
  // head_dim 64 it keeps M = 128, and its upper half is one region shared by
  // every V slot (the descriptor's leading byte offset points there), written
  // once: all zeros except dimension 64, which holds ones so that O^T row 64
  // accumulates the column sums of P.
  static constexpr int kVS = kKV;
  static constexpr bool kOnesRow = D == 64;
  static constexpr int kOnes = kOnesRow ? 16384 : 0;
  static constexpr int kQ = kHalves * NQP * 128;     // Q^T operand [half][NQP][128 B]
  static constexpr int kP = 2 * NQP * 128;           // P^T operand [kblock][NQP][128 B]
  static constexpr int kThreads = 384;               // 12 warps
  static constexpr int kCol = NQP < 32 ? 32 : NQP;   // tensor-memory columns per accumulator
  static constexpr uint32_t kTmemCols = 4 * kCol;    // S0, S1, O0, O1
  static constexpr int kOffV = KS * kKV;
  static constexpr int kOffOnes = kOffV + VS * kVS;  // 1024-byte aligned, like every tile
  static constexpr int kOffQ = kOffOnes + kOnes;
  static constexpr int kOffP = kOffQ + kQ;
  static constexpr int kOffBar = kOffP + 2 * kP;
  static constexpr int kNumBars = 2 * KS + 2 * VS + 4 * 2 + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  // misc: tmem slot, flag, votes[2][4], colmax[2][4][NQC], colsum[2][4][NQC], tlim[NQP],
  // rawrow[NQP], negated column references nref[2][NQC] (wide tiles, on the next 16-byte boundary)
  static constexpr bool kSmemMax = NQC > 32;
  static constexpr size_t kMisc = 16 + 32 + 4 * (18 * NQC + 2 * NQP) + (kSmemMax ? 16 : 0);
  static constexpr size_t kSmem = size_t(kOffMisc) + kMisc + 1024;
};

// Cluster-wide barrier of every thread (release / acquire): shared-memory
// writes before it, local or remote, are visible to every CTA after it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <int D, int NQP, int NQC, bool CAPTURE>
__global__ void __launch_bounds__(384, 1)
    verify_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap, const VerifyParams p) {
  using Cfg = TcCfg<D, NQP, NQC>;
  constexpr int KS = Cfg::KS;
  constexpr int VS = Cfg::VS;
  constexpr int kCol = Cfg::kCol;
  static_assert(D == 64 || D == 128, "head_dim");
  static_assert(NQP == 16 || NQP == 32 || NQP == 64, "MMA N");
  static_assert(NQC % 8 == 0 && NQC + (CAPTURE ? 2 : 0) <= NQP, "processed columns");
  static_assert(Cfg::kSmem <= 227 * 1024, "shared memory");

  griddep_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint8_t* qs = smem + Cfg::kOffQ;
  const uint32_t bar0 = sbase + Cfg::kOffBar;
  // barriers: K full/free (per K slot), V full/free (per V slot); S full, S
  // read, P ready, PV done (per softmax group); MMA drain
  auto kfull = [&](int s) { return bar0 + 8 * s; };
  auto kfree = [&](int s) { return bar0 + 8 * (KS + s); };
  auto vfull = [&](int s) { return bar0 + 8 * (2 * KS + s); };
  auto vfree = [&](int s) { return bar0 + 8 * (2 * KS + VS + s); };
  constexpr int B1 = 2 * KS + 2 * VS;
  auto sfull = [&](int g2) { return bar0 + 8 * (B1 + g2); };
  auto sread = [&](int g2) { return bar0 + 8 * (B1 + 2 + g2); };
  auto pready = [&](int g2) { return bar0 + 8 * (B1 + 4 + g2); };
  auto pvdone = [&](int g2) { return bar0 + 8 * (B1 + 6 + g2); };
  const uint32_t drain = bar0 + 8 * (B1 + 8);
  uint8_t* misc = smem + Cfg::kOffMisc;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
  int* flag = reinterpret_cast<int*>(misc + 4);
  int* votes = reinterpret_cast<int*>(misc + 16);                // [2][4]
  float* colmax = reinterpret_cast<float*>(misc + 48);           // [2][4][NQC]
  float* colsum = colmax + 8 * NQC;                              // [2][4][NQC]
  int* tlim = reinterpret_cast<int*>(colsum + 8 * NQC);          // [NQP]
  int* rawrow = tlim + NQP;                                      // [NQP] raw-logit row of a column, or -1
  float* mrun = reinterpret_cast<float*>(                        // [2][NQC] nref (wide tiles)
      (reinterpret_cast<uintptr_t>(rawrow + NQP) + 15) & ~uintptr_t(15));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int unit = b * p.hkv + g;
  const int T = p.gamma + 1;
  const int cap = p.max_pages * 16;

  if (tid == 0) {
    for (int s = 0; s < KS; ++s) {
      mbar_init(kfull(s), 1);
      mbar_init(kfree(s), 1);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(vfull(s), 1);
      mbar_init(vfree(s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(sfull(i), 1);
      mbar_init(sread(i), 128);
      mbar_init(pready(i), 128);
      mbar_init(pvdone(i), 1);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
    tmem_relinquish();
  }
  // Nothing above reads or writes global memory, so it overlaps the tail of
  // the previous kernel of the stream.
  griddep_wait();

  // Warps 1-9 request their chunks of the window queries first, so those
  // loads are in flight together with the context-length load below.
  constexpr int SN = 288;                      // threads of warps 1..9
  constexpr int CPR = D / 8;                   // 16-byte chunks per query row
  constexpr int QPER = (NQP * CPR + SN - 1) / SN;
  uint4 qreg[QPER];
#pragma unroll
  for (int u = 0; u < QPER; ++u) {
    const int i = tid - 32 + u * SN, n = i / CPR, c = i % CPR;
    qreg[u] = make_uint4(0, 0, 0, 0);
    if (warp >= 1 && warp <= 9 && i < NQP * CPR && n < p.nq) {
      const int t = n / p.group, hl = n - t * p.group;
      qreg[u] = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p.q) +
                                               ((size_t(b) * T + t) * p.hq + g * p.group + hl) * D)[c];
    }
  }
  // Producer roles (warps 0, 10, 11).  TMA issue rate is per warp, so a
  // tile's 32 boxes (8 pages x 2 column halves, of K and of V) are spread over
  // three warps, in half-warps:
  //   warp 0,  lanes 0-15:  K pages 0-5, arms the K slot's barrier;
  //   warp 10, lanes 0-15:  V pages 0-5, arms the V slot's barrier;
  //   warp 11, lanes 0-15:  K pages 6-7;  lanes 16-31: V pages 6-7.
  // Lane j < np of a half-warp loads page pf + j (two 64-column boxes).
  const int half = lane >> 4, hl = lane & 15;
  const unsigned hmask = 0xFFFFu << (16 * half);
  const bool producer = warp == 0 || warp >= 10;
  const bool active = producer && (warp == 11 || half == 0);
  const bool is_k = warp == 11 ? half == 0 : warp == 0;
  const bool arms = warp != 11;
  const int pf = warp == 11 ? 6 : 0, np = warp == 11 ? 2 : 6;
  // Clustered splits share the unit's pages evenly; workspace splits take
  // pages_per_split each (whole tiles).
  // (split * max_pages < 2^31: max_pages < 2^20, splits <= 128)
  const int pbeg = p.cluster_merge ? split * p.max_pages / p.num_splits
                                   : split * p.pages_per_split;
  const int pnext = p.cluster_merge ? (split + 1) * p.max_pages / p.num_splits
                                    : pbeg + p.pages_per_split;
  const int32_t* bt_row = p.block_table + size_t(b) * p.max_pages;
  // Block-table entries are prefetched four tiles ahead, one register per
  // tile modulo 4, so a load is consumed four iterations after its issue.
  // The loads do not wait for the context length: lane np of the half-warp
  // loads the tile's first page, which stands in for pages past the end of
  // the range (loaded again and masked by the softmax), and indices are
  // clamped to the row.
  auto table_entry = [&](int tt) {
    if (hl > np) return 0;
    const int page = pbeg + 8 * tt + (hl < np ? pf + hl : 0);
    return __ldg(&bt_row[min(page, p.max_pages - 1)]);
  };
  int held[4] = {0, 0, 0, 0};
  if (active) {
#pragma unroll
    for (int j = 0; j < 4; ++j) held[j] = table_entry(j);
  }

  int L = p.ctx_lens[b];
  if (L < 0 || L + T > cap) {
    if (tid == 0) set_error(p.err, kErrDeviceFault);
    L = max(0, min(L, cap - T));
  }
  const int npages = (L + T + 15) / 16;
  const int pend = min(pnext, npages);
  const int ntiles = pend > pbeg ? (pend - pbeg + 7) / 8 : 0;
  constexpr int cap0 = NQC;   // the summed captured query: MMA columns NQC and NQC + 1
  const int last_valid = L + p.gamma;

  __syncthreads();   // barriers initialised before anyone waits on them
  // Warps 0 and 10 start streaming K and V right away; warps 1-9 meanwhile
  // build the Q^T operand.
  uint32_t tmem = 0;
  if (warp >= 1 && warp <= 9) {
    const int st = tid - 32;
    // Q^T operand, K-major with the 128-byte swizzle: element (n, k) at
    // (k / 64) * NQP * 128 + n * 128 + (((k % 64) / 8) ^ (n % 8)) * 16 + (k % 8) * 2.
#pragma unroll
    for (int u = 0; u < QPER; ++u) {
      const int i = st + u * SN, n = i / CPR, c = i % CPR;
      if (i < NQP * CPR)
        *reinterpret_cast<uint4*>(qs + (c >> 3) * (NQP * 128) + n * 128 + (((c & 7) ^ (n & 7)) << 4)) =
            qreg[u];
    }
    if constexpr (Cfg::kOnesRow) {
      // the shared upper half of V^T: zeros, and ones at head dimension 64
      // (element (pos, 64) of the MN-major swizzled half sits at chunk pos % 8)
      for (int e = st; e < 128 * 8; e += SN) {
        const int pos = e / 8, ch = e % 8;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (ch == (pos & 7)) v.x = 0x3F80u;   // bf16 1.0 in the chunk's first element
        *reinterpret_cast<uint4*>(smem + Cfg::kOffOnes + pos * 128 + ch * 16) = v;
      }
    }
    for (int n = st; n < NQP; n += SN) {
      tlim[n] = n < p.nq ? min(n / p.group, p.gamma) : -1;
      if constexpr (!CAPTURE) {
        // raw-logit mode: column n = t * G + hl of a captured row t goes to row
        // (b * R + rank of t among the captured rows) * Hq + g * G + hl
        int rr = -1;
        if (p.raw && n < p.nq) {
          const int t = n / p.group, hl = n - t * p.group;
          if ((p.row_mask >> t) & 1u)
            rr = (b * p.raw_rows + __popc(p.row_mask & ((1u << t) - 1u))) * p.hq + g * p.group + hl;
        }
        rawrow[n] = rr;
      }
    }
    if (CAPTURE) {
      named_bar(4, SN);
      // the summed captured query as a bf16 part and a bf16 remainder, summed
      // from the Q tile just written (rows t * G .. t * G + G - 1 of each row t)
      auto qoff = [&](int n, int k) {
        return (k >> 6) * (NQP * 128) + n * 128 + ((((k & 63) >> 3) ^ (n & 7)) << 4) + (k & 7) * 2;
      };
      for (int j = st; j < D; j += SN) {
        float acc = 0.f;
        for (int t = 0; t <= p.gamma; ++t) {
          if (!((p.row_mask >> t) & 1u)) continue;
          for (int hl = 0; hl < p.group; ++hl)
            acc += __bfloat162float(
                *reinterpret_cast<const __nv_bfloat16*>(qs + qoff(t * p.group + hl, j)));
        }
        const __nv_bfloat16 hi = __float2bfloat16_rn(acc);
        const __nv_bfloat16 lo = __float2bfloat16_rn(acc - __bfloat162float(hi));
        *reinterpret_cast<__nv_bfloat16*>(qs + qoff(cap0, j)) = hi;
        *reinterpret_cast<__nv_bfloat16*>(qs + qoff(cap0 + 1, j)) = lo;
      }
    }
    // Generic-proxy writes of Q must be visible to the tensor cores (async proxy).
    fence_proxy_async_smem();
    tc_fence_before();
    named_bar(4, SN);
    tc_fence_after();
    tmem = *tmem_slot;
  }
  bool ok = true;
  // A softmax group's final partial state for head dimension i: O^T row i
  // (unnormalised), and column i's running maximum and row sum (i < NQC).
  float o[NQC];
  float Mg = kEmptyMax, Lg = 0.f;
  const bool on_chip = p.cluster_merge || p.num_splits == 1;

  if (warp == 0 || warp >= 10) {
    // ------------------------------------------------------------ producers
    // (roles and the first block-table entries: above)
    const int depth = is_k ? KS : VS;
    const CUtensorMap* map = is_k ? &kmap : &vmap;
    const uint32_t ring = sbase + (is_k ? 0 : Cfg::kOffV);
    const uint32_t slot_bytes = is_k ? Cfg::kKV : Cfg::kVS;
    // The cache is streamed once per pass: its lines leave L2 first, so the
    // scores, queries and block table stay there for the kernels after this.
    const uint64_t stream_pol = l2_evict_first_policy();
    int issued = 0;
    if (active) {
      for (int t0 = 0; t0 < ntiles && ok; t0 += 4) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int t = t0 + j;
          if (t >= ntiles) break;
          const int s = t % depth;
          const uint32_t full = is_k ? kfull(s) : vfull(s);
          const uint32_t freed = is_k ? kfree(s) : vfree(s);
          // the half-warp agrees on the outcome, so it leaves together
          if (t >= depth &&
              !__all_sync(hmask, mbar_wait_bounded(freed, ((t / depth) - 1) & 1))) {
            ok = false;
            break;
          }
          int phys = held[j];
          const int first = __shfl_sync(hmask, phys, np, 16);
          if (pbeg + 8 * t + pf + hl >= pend) phys = first;
          held[j] = table_entry(t + 4);
          if (hl < np && (phys < 0 || phys >= p.num_pages)) {
            set_error(p.err, kErrDeviceFault);
            phys = 0;
          }
          // one arrival per phase, with the whole tile's bytes; the other
          // half-warp's loads count against it
          if (arms && hl == 0) mbar_arrive_expect_tx(full, Cfg::kKV);
          __syncwarp(hmask);
          if (hl < np) {
            const int row = (phys * p.hkv + g) * 16;
            const uint32_t dst = ring + s * slot_bytes + (pf + hl) * 2048;
            tma_load_2d_hint(dst, map, 0, row, full, stream_pol);
            if constexpr (D == 128) tma_load_2d_hint(dst + 16384, map, 64, row, full, stream_pol);
          }
          __syncwarp(hmask);
          issued = t + 1;
        }
      }
      if (!ok) {
        if (hl == 0) set_error(p.err, kErrDeviceTimeout);
        for (int t = max(0, issued - depth); t < issued; ++t)
          (void)mbar_wait_bounded(is_k ? kfull(t % depth) : vfull(t % depth), (t / depth) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop, so its control flow and the operand
    // descriptors stay warp-uniform; one elected lane issues and commits.
    constexpr uint32_t idS = idesc_bf16(128, NQP, 0, 0);
    // M = 128 dims (padded at D = 64); P^T is MN-major (one 128-byte row of
    // 64 columns per position) when NQP = 64, else K-major
    constexpr bool kPmn = NQP == 64;
    constexpr uint32_t idPV = idesc_bf16(128, NQP, 1, kPmn ? 1 : 0);
    const bool leader = elect_one();
    // Descriptors without their start address; the address field (bits 0-13)
    // holds (address / 16) mod 2^14, the part of a shared-window address the
    // tensor cores use, so it is added and masked last.
    const uint64_t dSw = smem_desc(0, 16, 1024, 2);       // K-major, 128-byte swizzle
    const uint64_t dVmn = smem_desc(0, 16384, 1024, 2);   // MN-major operand, halves 16 KB apart
    auto with_addr = [](uint64_t d, uint32_t a16) { return d | uint64_t(a16 & 0x3FFFu); };
    const uint32_t qb = (sbase + Cfg::kOffQ) >> 4;
    auto wait_all = [&](uint32_t bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity));
    };
    auto issue_pv = [&](int t) -> bool {
      const int gg = t & 1, s = t % VS;
      if (!wait_all(pready(gg), (t >> 1) & 1)) return false;
      if (!wait_all(vfull(s), (t / VS) & 1)) return false;
      tc_fence_after();
      const uint32_t vb = (sbase + Cfg::kOffV + s * Cfg::kVS) >> 4;
      const uint32_t pb = (sbase + Cfg::kOffP + gg * Cfg::kP) >> 4;
      // V^T as the MN-major A operand; at head_dim 64 its upper half is the
      // shared ones region, one leading byte offset past the slot
      const uint64_t dV =
          Cfg::kOnesRow ? smem_desc(0, uint32_t(Cfg::kOffOnes - Cfg::kOffV - s * Cfg::kVS), 1024, 2)
                        : dVmn;
      if (leader) {
#pragma unroll
        for (int kp = 0; kp < 8; ++kp)
          tc_mma(tmem + 2 * kCol + kCol * gg, with_addr(dV, vb + kp * 128),
                 kPmn ? with_addr(dVmn, pb + kp * 128)
                      : with_addr(dSw, pb + (kp >> 2) * (NQP * 8) + (kp & 3) * 2),
                 idPV, t >= 2 || kp > 0);
        tc_commit(pvdone(gg));
        tc_commit(vfree(s));
      }
      __syncwarp();
      return true;
    };
    for (int t = 0; t < ntiles && ok; ++t) {
      const int s = t % KS, gg = t & 1;
      if (!wait_all(kfull(s), (t / KS) & 1)) { ok = false; break; }
      if (t >= 2 && !wait_all(sread(gg), ((t >> 1) - 1) & 1)) { ok = false; break; }
      tc_fence_after();
      const uint32_t kb = (sbase + s * Cfg::kKV) >> 4;
      if (leader) {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          tc_mma(tmem + kCol * gg, with_addr(dSw, kb + (ks >> 2) * 1024 + (ks & 3) * 2),
                 with_addr(dSw, qb + (ks >> 2) * (NQP * 8) + (ks & 3) * 2), idS, ks > 0);
        tc_commit(sfull(gg));
        tc_commit(kfree(s));
      }
      __syncwarp();
      if (t >= 1 && !issue_pv(t - 1)) { ok = false; break; }
    }
    if (ok && ntiles > 0 && !issue_pv(ntiles - 1)) ok = false;
    if (!ok && leader) set_error(p.err, kErrDeviceTimeout);
    // every MMA issued has completed before tensor memory is released
    if (leader) tc_commit(drain);
    __syncwarp();
    (void)mbar_wait_bounded(drain, 0);
  } else {
    // ------------------------------------------------------------ softmax groups (warps 2-9)
    const int grp = (warp - 2) >> 2;          // 0: even tiles, 1: odd tiles
    const int q4 = warp & 3;                  // tensor-memory lane quarter of this warp
    const int i = 32 * q4 + lane;             // tile position / head dimension owned
    const uint32_t tl = tmem + (uint32_t(32 * q4) << 16);
    const uint32_t s_col = kCol * grp, o_col = 2 * kCol + kCol * grp;
    // Narrow tiles (at most 32 columns) keep each column's running maximum m
    // in registers and take P = 2^(x * scale_log2 - m).  Wide tiles, where the
    // softmax's instruction count sets the pace, keep per column a reference r
    // (m, or 0 while the column has seen no unmasked logit: m = kEmptyMax) as
    // -r in the group's nref row of shared memory, read as 16-byte vectors,
    // and take y = x * scale_log2 - r in one FMA, so that P = 2^y needs no
    // other per-element step and the rescale test is the largest y against
    // the slack; `empty` flags the columns still without a maximum (identical
    // in every thread of the group).  Row sums per column and thread are kept
    // unless V's ones row makes the PV MMA accumulate them.
    constexpr bool kOffset = Cfg::kSmemMax;
    float m[kOffset ? 1 : NQC], ls[Cfg::kOnesRow ? 1 : NQC];
#pragma unroll
    for (int n = 0; n < NQC; ++n) {
      if constexpr (!kOffset) m[n] = kEmptyMax;
      if constexpr (!Cfg::kOnesRow) ls[n] = 0.f;
    }
    float* nrg = mrun + grp * NQC;
    if constexpr (kOffset) {
      if (i < NQC) nrg[i] = 0.f;
      named_bar(1 + grp, 128);
    }
    uint64_t empty = NQC == 64 ? ~0ull : (1ull << NQC) - 1;
    // Columns nq .. NQC - 1 multiply zero query rows: their logits are 0 and
    // nothing reads their output.
    float* srow = CAPTURE ? p.scores + size_t(unit) * p.score_stride : nullptr;
    int Lcap = L;
    if (CAPTURE && L > p.score_stride) {
      if (i == 0 && grp == 0) set_error(p.err, kErrDeviceFault);
      Lcap = p.score_stride;
    }
    int mytiles = 0;
    // A failed (timed-out) wait is carried to the group vote below, so the 128
    // threads of a group always leave the loop together.
    for (int t = grp; t < ntiles; t += 2) {
      const int k = t >> 1, s = t % VS;
      bool okt = ok && mbar_wait_bounded(sfull(grp), k & 1);
      tc_fence_after();
      const int page = pbeg + 8 * t + (i >> 4);
      const bool live = page < pend;
      const int pos = page * 16 + (i & 15);
      float y[NQC];
      float cx[2] = {0.f, 0.f};   // the two capture columns
#pragma unroll
      for (int n = 0; n < NQC; ++n) y[n] = 0.f;
      if (okt) {
#pragma unroll
        for (int c = 0; c < NQC / 8; ++c) {
          float v8[8];
          tmem_ld8(tl + s_col + 8 * c, v8);
#pragma unroll
          for (int e = 0; e < 8; ++e) y[8 * c + e] = v8[e];
        }
        if constexpr (CAPTURE) tmem_ld2(tl + s_col + cap0, cx);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(sread(grp));
      }
      if (CAPTURE && okt && live && pos < Lcap) srow[pos] = (cx[0] + cx[1]) * p.scale;
      if (!CAPTURE && p.raw && okt && live && pos < min(L, p.raw_stride)) {
        // the pages' way: every captured row's logit of every head goes to memory
#pragma unroll
        for (int n = 0; n < NQC; ++n) {
          const int rr = rawrow[n];
          if (rr >= 0) p.raw[size_t(rr) * p.raw_stride + pos] = y[n] * p.scale;
        }
      }
      // logits in log2 units (less the reference, wide tiles); positions past
      // the split's range, and window positions a row may not see yet
      // (pos > L + t), are masked
      bool need = false;
      if constexpr (kOffset) {
        const float4* nr4 = reinterpret_cast<const float4*>(nrg);
#pragma unroll
        for (int c = 0; c < NQC / 4; ++c) {
          const float4 v = nr4[c];
          y[4 * c + 0] = fmaf(y[4 * c + 0], p.scale_log2, v.x);
          y[4 * c + 1] = fmaf(y[4 * c + 1], p.scale_log2, v.y);
          y[4 * c + 2] = fmaf(y[4 * c + 2], p.scale_log2, v.z);
          y[4 * c + 3] = fmaf(y[4 * c + 3], p.scale_log2, v.w);
        }
        if (!live || pos > L) {
#pragma unroll
          for (int n = 0; n < NQC; ++n)
            if (!live || pos > L + tlim[n]) y[n] = -INFINITY;
        }
        float ym[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int n = 0; n < NQC; ++n) ym[n & 3] = fmaxf(ym[n & 3], y[n]);
        need = fmaxf(fmaxf(ym[0], ym[1]), fmaxf(ym[2], ym[3])) > kRescaleSlack;
      } else {
        const float sl2 = live ? p.scale_log2 : 0.f;
        const float bias = live ? 0.f : -INFINITY;
#pragma unroll
        for (int n = 0; n < NQC; ++n) y[n] = fmaf(y[n], sl2, bias);
        if (pos > L) {
#pragma unroll
          for (int n = 0; n < NQC; ++n)
            if (pos > L + tlim[n]) y[n] = -INFINITY;
        }
#pragma unroll
        for (int n = 0; n < NQC; ++n) need |= y[n] > m[n] + kRescaleSlack;
      }
      const int lpos = (live ? page : pbeg + 8 * t) * 16 + (i & 15);   // position loaded in row i
      if (okt && lpos > last_valid) {
        // a cache slot past the window: zero its V row so 0 * garbage cannot be NaN
        okt = mbar_wait_bounded(vfull(s), (t / VS) & 1);
        uint8_t* vrow = smem + Cfg::kOffV + s * Cfg::kVS + i * 128;
        if (okt) {
#pragma unroll
          for (int h = 0; h < Cfg::kHalves; ++h)
#pragma unroll
            for (int cc = 0; cc < 8; ++cc)
              *reinterpret_cast<uint4*>(vrow + h * 16384 + ((cc ^ (i & 7)) << 4)) =
                  make_uint4(0, 0, 0, 0);
        }
      }
      const int wvote = (__any_sync(0xffffffffu, need) ? 1 : 0) | (__any_sync(0xffffffffu, !okt) ? 2 : 0);
      if (lane == 0) votes[grp * 4 + q4] = wvote;
      named_bar(1 + grp, 128);
      const int allv = votes[grp * 4] | votes[grp * 4 + 1] | votes[grp * 4 + 2] | votes[grp * 4 + 3];
      if (allv & 2) {
        ok = false;
        break;
      }
      // The group's previous PV (tile t - 2) must have finished before its O^T
      // is rescaled or its P^T buffer rewritten.
      bool pv_ok = k == 0 || mbar_wait_bounded(pvdone(grp), (k - 1) & 1);
      tc_fence_after();
      if ((allv & 1) || (kOffset && empty)) {
        // column maxima over the group's 128 positions
#pragma unroll
        for (int n = 0; n < NQC; ++n) {
          float v = y[n];
#pragma unroll
          for (int o2 = 16; o2 > 0; o2 >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o2));
          if (lane == 0) colmax[(grp * 4 + q4) * NQC + n] = v;
        }
        named_bar(1 + grp, 128);
        const float* cm = colmax + grp * 4 * NQC;
        auto cmax = [&](int n) {
          return fmaxf(fmaxf(cm[n], cm[NQC + n]), fmaxf(cm[2 * NQC + n], cm[3 * NQC + n]));
        };
        // Per 8-column chunk: the new maximum m', the factor 2^(m - m') for
        // O^T and the row sums and (wide tiles) the new reference r', with y
        // shifted to it.
        uint64_t empty2 = empty;
#pragma unroll
        for (int c = 0; c < NQC / 8; ++c) {
          float f8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int n = 8 * c + e;
            if constexpr (kOffset) {
              const float nro = nrg[n];
              const float mold = ((empty >> n) & 1) ? kEmptyMax : -nro;
              const float mnew = fmaxf(mold, cmax(n) - nro);
              const bool now_empty = mnew == kEmptyMax;
              f8[e] = ex2(mold - mnew);
              if (!now_empty) empty2 &= ~(1ull << n);
              y[n] += (now_empty ? 0.f : -mnew) - nro;
            } else {
              const float mnew = fmaxf(m[n], cmax(n));
              f8[e] = ex2(m[n] - mnew);
              m[n] = mnew;
            }
            if constexpr (!Cfg::kOnesRow) ls[n] *= f8[e];
          }
          if (k > 0 && pv_ok) {
            float v8[8];
            tmem_ld8(tl + o_col + 8 * c, v8);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 8; ++e) v8[e] *= f8[e];
            tmem_st8(tl + o_col + 8 * c, v8);
          }
        }
        if (k > 0 && pv_ok) tmem_st_wait();
        named_bar(1 + grp, 128);   // colmax (and nref) read; colmax is rewritten at the next rescale
        if constexpr (kOffset) {
          if (i < NQC) {
            const float nro = nrg[i];
            const float mold = ((empty >> i) & 1) ? kEmptyMax : -nro;
            const float mnew = fmaxf(mold, cmax(i) - nro);
            nrg[i] = mnew == kEmptyMax ? 0.f : -mnew;
          }
          named_bar(1 + grp, 128);   // new references visible
          empty = empty2;
        }
      }
      // P = 2^y (wide tiles) or 2^(y - m)
      auto pcol = [&](int n) {
        if constexpr (kOffset)
          return ex2(y[n]);
        else
          return ex2(y[n] - m[n]);
      };
      if constexpr (NQP == 64) {
        // P^T MN-major: position i's row of 64 columns, eight 16-byte chunks
        // (eight bf16 columns each, one store per chunk), chunk c at c ^ (i % 8)
        // (128-byte swizzle); columns past NQC are 0
        uint8_t* prow = smem + Cfg::kOffP + grp * Cfg::kP + i * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t w4[4] = {0u, 0u, 0u, 0u};
          if (8 * c < NQC) {
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              const int n = 8 * c + e;
              const float p0 = pcol(n), p1 = pcol(n + 1);
              if constexpr (!Cfg::kOnesRow) {
                ls[n] += p0;
                ls[n + 1] += p1;
              }
              w4[e / 2] = pack_bf16x2(p0, p1);
            }
          }
          *reinterpret_cast<uint4*>(prow + ((c ^ (i & 7)) << 4)) =
              make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
      } else {
        // P^T K-major: element (n, i) at (i / 64) * NQP * 128 + n * 128 +
        // (((i % 64) / 8) ^ (n % 8)) * 16 + (i % 8) * 2 (128-byte swizzle)
        uint8_t* pbuf = smem + Cfg::kOffP + grp * Cfg::kP + (i >> 6) * (NQP * 128) + (i & 7) * 2;
        const int ci = (i & 63) >> 3;
#pragma unroll
        for (int n = 0; n < NQC; ++n) {
          const float pv = pcol(n);
          if constexpr (!Cfg::kOnesRow) ls[n] += pv;
          *reinterpret_cast<__nv_bfloat16*>(pbuf + n * 128 + ((ci ^ (n & 7)) << 4)) =
              __float2bfloat16_rn(pv);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(pready(grp));
      if (!pv_ok) ok = false;   // the group leaves at the next vote
      mytiles = k + 1;
    }
    // The group's last PV completes its O^T.
    if (mytiles > 0 && !mbar_wait_bounded(pvdone(grp), (mytiles - 1) & 1)) ok = false;
    tc_fence_after();
    if (!ok && i == 0) set_error(p.err, kErrDeviceTimeout);

    // Each group's (m, l, O^T) is a partial state of its own, merged together
    // with the splits' states, so no group waits on the other's arithmetic.
    // Row sums over the group's 128 positions:
    if constexpr (!Cfg::kOnesRow) {
#pragma unroll
      for (int n = 0; n < NQC; ++n) {
        float v = ls[n];
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o2);
        if (lane == 0) colsum[(grp * 4 + q4) * NQC + n] = v;
      }
    }
    // this thread's O^T row (head dimension i), unnormalised
#pragma unroll
    for (int n = 0; n < NQC; ++n) o[n] = 0.f;
    if (mytiles > 0) {
#pragma unroll
      for (int c = 0; c < NQC / 8; ++c) {
        float v8[8];
        tmem_ld8(tl + o_col + 8 * c, v8);
#pragma unroll
        for (int e = 0; e < 8; ++e) o[8 * c + e] = v8[e];
      }
      tmem_ld_wait();
    }
    if constexpr (Cfg::kOnesRow) {
      // O^T row 64 accumulated the column sums of P (V's ones row)
      if (i == 64) {
#pragma unroll
        for (int n = 0; n < NQC; ++n) colsum[grp * 4 * NQC + n] = o[n];
      }
    }
    named_bar(1 + grp, 128);
    if (i < NQC) {
      const float* cs = colsum + grp * 4 * NQC;
      if (mytiles > 0)
        Lg = Cfg::kOnesRow ? cs[i] : cs[i] + cs[NQC + i] + cs[2 * NQC + i] + cs[3 * NQC + i];
      if constexpr (kOffset) {
        Mg = ((empty >> i) & 1) ? kEmptyMax : -nrg[i];
      } else {
#pragma unroll
        for (int n = 0; n < NQC; ++n)
          if (n == i) Mg = m[n];
      }
    }
    if (!on_chip) {
      // partial 2 * split + grp of the unit's 2 * num_splits
      const size_t part = (size_t(unit) * p.num_splits + split) * 2 + grp;
#pragma unroll
      for (int n = 0; n < NQC; ++n)
        if (n < p.nq && i < D) p.part_o[(part * p.nq + n) * D + i] = o[n];
      if (i < p.nq) {
        p.part_ml[(part * p.nq + i) * 2 + 0] = Mg;
        p.part_ml[(part * p.nq + i) * 2 + 1] = Lg;
      }
    }
  }

  // Every CTA of the cluster is past its last MMA and holds no load in flight,
  // so its K ring is free from here on.
  tc_fence_before();
  if (on_chip)
    cluster_sync_all();
  else
    __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
  auto out_row = [&](int n) {
    const int t = n / p.group, hl2 = n - t * p.group;
    return out + ((size_t(b) * T + t) * p.hq + g * p.group + hl2) * D;
  };
  if (on_chip) {
    // Split-KV merge on chip (one split: a cluster of one CTA).  Row n of the
    // output belongs to cluster rank n % S, which receives in its K ring, at
    // slot n / S, the 2S partial states of the row (state 2 * rank + group of
    // each sender, O[D] then m and l), pushed with distributed-shared-memory
    // stores; one cluster barrier publishes them and each rank merges its rows
    // from local shared memory: O = sum_q 2^(m_q - M) O_q / sum_q 2^(m_q - M) l_q
    // with M = max_q m_q.  Nothing reads another CTA's shared memory, so no
    // barrier precedes the exit.
    constexpr int RS = D + 4;   // one received state: O[D], m, l, padding to 16 bytes
    static_assert(2 * (NQC + kMaxVerifyCluster) * RS * 4 <= KS * Cfg::kKV, "receive area");
    static_assert(2 * kMaxVerifyCluster <= 32, "one lane per state in the weight pass");
    cg::cluster_group cluster = cg::this_cluster();
    const int S = p.cluster_merge ? p.cluster_size : 1, r = (int)cluster.block_rank();
    const int C = p.num_splits / S, c = split / S;   // clusters of the unit, this one's index
    const float* recv = reinterpret_cast<const float*>(smem);
    if (warp >= 2 && warp <= 9) {
      const int grp = (warp - 2) >> 2, i = 32 * (warp & 3) + lane;
      const int q = 2 * r + grp;
      int owner = 0, slot = 0;
#pragma unroll
      for (int n = 0; n < NQC; ++n) {
        if (n < p.nq && i < D)
          st_cluster_f32(cluster_map(sbase + 4 * ((slot * 2 * S + q) * RS + i), owner), o[n]);
        if (++owner == S) {
          owner = 0;
          ++slot;
        }
      }
      if (i < p.nq) {
        const uint32_t dst = cluster_map(sbase + 4 * (((i / S) * 2 * S + q) * RS + D), i % S);
        st_cluster_f32(dst, Mg);
        st_cluster_f32(dst + 4, Lg);
      }
    }
    cluster_sync_all();
    const int nown = r < p.nq ? (p.nq - r + S - 1) / S : 0;
    // Weights 2^(m_q - M) / sum_q' 2^(m_q' - M) l_q' of the 2S states of each
    // owned row (one warp per row, lane q), into the free V ring, with the
    // row's cluster-level maximum M and sum (used when C > 1) ...
    // (nown <= NQC <= 64 rows, 2S <= 32 states, C <= 32 clusters)
    static_assert((64 * 2 * kMaxVerifyCluster + 2 * 64 + 64 * 32) * 4 <= VS * Cfg::kVS,
                  "merge weights fit the V ring");
    float* wts = reinterpret_cast<float*>(smem + Cfg::kOffV);   // [nown][2S]
    float* rowml = wts + 64 * 2 * kMaxVerifyCluster;           // [nown][2]
    for (int k = warp; k < nown; k += Cfg::kThreads / 32) {
      const float* st = recv + k * 2 * S * RS;
      const bool has = lane < 2 * S;
      const float m = has ? st[lane * RS + D] : kEmptyMax;
      const float l = has ? st[lane * RS + D + 1] : 0.f;
      float M = m;
#pragma unroll
      for (int o2 = 16; o2 > 0; o2 >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o2));
      const float f = has ? ex2(m - M) : 0.f;
      float Lsum = f * l;
#pragma unroll
      for (int o2 = 16; o2 > 0; o2 >>= 1) Lsum += __shfl_xor_sync(0xffffffffu, Lsum, o2);
      if (has) wts[k * 2 * S + lane] = Lsum > 0.f ? f / Lsum : 0.f;
      if (lane == 0) {
        rowml[2 * k] = M;
        rowml[2 * k + 1] = Lsum;
      }
    }
    __syncthreads();
    // ... then four output elements per thread: sum_q w_q O_q[d .. d + 3]
    for (int e = tid; e < nown * (D / 4); e += Cfg::kThreads) {
      const int k = e / (D / 4), d = 4 * (e - k * (D / 4));
      const float* st = recv + k * 2 * S * RS + d;
      const float* wk = wts + k * 2 * S;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
      for (int q = 0; q < 2 * S; ++q) {
        const float4 v = *reinterpret_cast<const float4*>(st + q * RS);
        const float wq = wk[q];
        acc.x += wq * v.x;
        acc.y += wq * v.y;
        acc.z += wq * v.z;
        acc.w += wq * v.w;
      }
      if (C == 1) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 pk;
        pk.x = *reinterpret_cast<const uint32_t*>(&lo);
        pk.y = *reinterpret_cast<const uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(out_row(r + k * S) + d) = pk;
      } else {
        // this cluster's normalised row, merged across the unit's clusters below
        const size_t row = (size_t(unit) * C + c) * p.nq + (r + k * S);
        *reinterpret_cast<float4*>(p.part_o + row * D + d) = acc;
      }
    }
    if (C > 1) {
      // Cross-cluster merge through the workspace, per owner rank: rank r of
      // every cluster of the unit writes its rows' (o_c, M_c, L_c), takes the
      // ticket of (unit, r), and the last to arrive combines them:
      // out = sum_c F_c o_c / sum_c F_c with F_c = 2^(M_c - max M) L_c.
      for (int k = tid; k < nown; k += Cfg::kThreads) {
        const size_t row = (size_t(unit) * C + c) * p.nq + (r + k * S);
        p.part_ml[2 * row] = rowml[2 * k];
        p.part_ml[2 * row + 1] = rowml[2 * k + 1];
      }
      __threadfence();
      __syncthreads();
      if (tid == 0) *flag = atomicAdd(&p.tickets[unit * S + r], 1) == C - 1;
      __syncthreads();
      if (*flag) {
        __threadfence();
        float* w2 = rowml + 2 * 64;   // [nown][C]
        for (int k = warp; k < nown; k += Cfg::kThreads / 32) {
          const bool has = lane < C;
          const size_t row = (size_t(unit) * C + lane) * p.nq + (r + k * S);
          const float m = has ? __ldcg(&p.part_ml[2 * row]) : kEmptyMax;
          const float l = has ? __ldcg(&p.part_ml[2 * row + 1]) : 0.f;
          float M = m;
#pragma unroll
          for (int o2 = 16; o2 > 0; o2 >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o2));
          const float F = has ? ex2(m - M) * l : 0.f;
          float Fs = F;
#pragma unroll
          for (int o2 = 16; o2 > 0; o2 >>= 1) Fs += __shfl_xor_sync(0xffffffffu, Fs, o2);
          if (has) w2[k * C + lane] = Fs > 0.f ? F / Fs : 0.f;
        }
        __syncthreads();
        for (int e = tid; e < nown * (D / 4); e += Cfg::kThreads) {
          const int k = e / (D / 4), d = 4 * (e - k * (D / 4));
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int q = 0; q < C; ++q) {
            const size_t row = (size_t(unit) * C + q) * p.nq + (r + k * S);
            const float4 v = __ldcg(reinterpret_cast<const float4*>(p.part_o + row * D + d));
            const float wq = w2[k * C + q];
            acc.x += wq * v.x;
            acc.y += wq * v.y;
            acc.z += wq * v.z;
            acc.w += wq * v.w;
          }
          const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
          const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
          uint2 pk;
          pk.x = *reinterpret_cast<const uint32_t*>(&lo);
          pk.y = *reinterpret_cast<const uint32_t*>(&hi);
          *reinterpret_cast<uint2*>(out_row(r + k * S) + d) = pk;
        }
        if (tid == 0) p.tickets[unit * S + r] = 0;
      }
    }
  } else {
    SplitWorkspace ws{p.tickets, p.part_ml, p.part_o};
    finish_splits<D, Cfg::kThreads, NQC>(ws, unit, p.num_splits, 2 * p.num_splits, p.nq, out_row,
                                         reinterpret_cast<float*>(smem), flag);
  }
}

template <int D, int NQP, int NQC, bool CAP>
static cudaError_t configure_tc() {
  using Cfg = TcCfg<D, NQP, NQC>;
  static std::atomic<uint32_t> configured{0};
  return once_per_device(configured, [] {
    cudaError_t e = cudaFuncSetAttribute(verify_tc_kernel<D, NQP, NQC, CAP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)Cfg::kSmem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(verify_tc_kernel<D, NQP, NQC, CAP>,
                                cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  });
}

// Launch (launch = true) or, with launch = false, the number of clusters of
// p.cluster_size CTAs that can be resident at once (into *clusters).
template <int D, int NQP, int NQC, bool CAP>
static cudaError_t launch_tc(const CUtensorMap& kmap, const CUtensorMap& vmap,
                             const VerifyParams& p, int batch, cudaStream_t stream, bool launch,
                             int* clusters) {
  using Cfg = TcCfg<D, NQP, NQC>;
  cudaError_t e = configure_tc<D, NQP, NQC, CAP>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.num_splits, p.hkv, batch);
  cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
  cfg.dynamicSmemBytes = Cfg::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.cluster_merge ? p.cluster_size : 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = launch ? 2 : 1;
  if (!launch)
    return cudaOccupancyMaxActiveClusters(clusters, verify_tc_kernel<D, NQP, NQC, CAP>, &cfg);
  return cudaLaunchKernelEx(&cfg, verify_tc_kernel<D, NQP, NQC, CAP>, kmap, vmap, p);
}

// The softmax's columns NQC = nq rounded up to 8, and the MMA width NQP (with
// capture the two summed-query columns NQC, NQC + 1 come on top).
template <int D, bool CAP>
static cudaError_t launch_tc_cols(const CUtensorMap& kmap, const CUtensorMap& vmap,
                                  const VerifyParams& p, int batch, cudaStream_t s, bool launch,
                                  int* clusters) {
  if (!verify_tc_supported(D, p.nq, CAP)) return cudaErrorInvalidValue;
  const int nqc = (p.nq + 7) / 8 * 8, nqp = verify_tc_mma_columns(p.nq, CAP);
#define VEGAS_TC_CASE(P_, C_)                                                    \
  if constexpr (C_ + (CAP ? 2 : 0) <= P_)                                        \
    if (nqp == P_ && nqc == C_)                                                  \
      return launch_tc<D, P_, C_, CAP>(kmap, vmap, p, batch, s, launch, clusters);
  VEGAS_TC_CASE(16, 8)
  VEGAS_TC_CASE(16, 16)
  VEGAS_TC_CASE(32, 16)
  VEGAS_TC_CASE(32, 24)
  VEGAS_TC_CASE(32, 32)
  VEGAS_TC_CASE(64, 32)
  VEGAS_TC_CASE(64, 40)
  if constexpr (D == 64) {
    VEGAS_TC_CASE(64, 48)
    VEGAS_TC_CASE(64, 56)
    VEGAS_TC_CASE(64, 64)
  }
#undef VEGAS_TC_CASE
  return cudaErrorInvalidValue;
}

#define VEGAS_CAT2(a, b) a##b
#define VEGAS_CAT(a, b) VEGAS_CAT2(a, b)

cudaError_t VEGAS_CAT(launch_verify_tc_d, VEGAS_TC_D)(const CUtensorMap& kmap,
                                                     const CUtensorMap& vmap,
                                                     const VerifyParams& p, bool capture,
                                                     int batch, cudaStream_t stream) {
  constexpr int D = VEGAS_TC_D;
  return capture ? launch_tc_cols<D, true>(kmap, vmap, p, batch, stream, true, nullptr)
                 : launch_tc_cols<D, false>(kmap, vmap, p, batch, stream, true, nullptr);
}

int VEGAS_CAT(verify_tc_max_active_clusters_d, VEGAS_TC_D)(int nq, bool capture, int cluster) {
  constexpr int D = VEGAS_TC_D;
  if (cluster < 1 || cluster > kMaxVerifyCluster) return 0;
  if (!verify_tc_supported(D, nq, capture)) return 0;
  constexpr int kDevices = 32;
  // [device][capture][column tiles of the softmax][cluster]: 0 unknown, -1 none, else the count
  static std::atomic<int> cache[kDevices][2][9][kMaxVerifyCluster + 1];
  const int ct = (nq + 7) / 8;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevices) return 0;
  std::atomic<int>& slot = cache[dev][capture ? 1 : 0][ct][cluster];
  int c = slot.load(std::memory_order_acquire);
  if (c == 0) {
    VerifyParams p{};
    p.hkv = 1;
    p.nq = nq;
    p.num_splits = cluster;
    p.cluster_size = cluster;
    p.cluster_merge = 1;
    CUtensorMap none{};
    int n = 0;
    cudaError_t e = capture ? launch_tc_cols<D, true>(none, none, p, 1, 0, false, &n)
                            : launch_tc_cols<D, false>(none, none, p, 1, 0, false, &n);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();
      n = 0;
    }
    c = n > 0 ? n : -1;
    slot.store(c, std::memory_order_release);
  }
  return c > 0 ? c : 0;
}

}  // namespace vegas
