// Verify attention with fused Collect-2-Query logit capture.
//
// "Vegas: Self-Speculative Decoding with Verification-Guided Sparse
// Attention", gist.science technical summary: §2 "Core mechanism" (the verify
// phase runs full attention and thereby computes every KV entry's logits),
// §2.A (the selection objective sums the logits over draft rows and the query
// heads of the group), §2.B "Collect-2-Query" (only two rows are collected),
// §3 "Implementation" (logits taken before softmax normalisation).
//
// Grid (num_splits, Hkv, B): one CTA per (split of the KV pages, KV head,
// sequence).  Each warp walks its own steps of P consecutive pages (step w,
// w+W, ...) through a private ring of TMA stages; a stage holds P pages of K
// and of V, loaded with 2-D tensor TMA (128-byte swizzle) straight from the
// paged cache, one mbarrier per stage.  The warp computes S^T for all
// (gamma+1)*G query rows of the unit at once (positions x query rows) with
// mma.sync, runs the lazy online softmax and O^T += V^T P^T.  Warp states merge
// in shared memory, splits merge through the workspace (last-arriving CTA).
//
// Capture.  The captured score of position i is
//   s_i = sum_{t in rows} sum_{h in group} (q_th . k_i) * scale
//       = (sum_{t,h} q_th) . k_i * scale,
// so the kernel adds the summed captured query as two extra query columns --
// its bf16 rounding and the bf16 rounding of the remainder -- and the score is
// the sum of those two columns of the same S^T tile, times the scale.  The
// two columns take no part in the softmax.
#include "kernels.h"
#include "split_merge.cuh"

namespace vegas {

template <int D, int NT>
struct VerifyCfg {
  static constexpr bool kQSmem = (D == 128) ? NT >= 4 : NT >= 7;   // Q^T fragments in smem
  static constexpr int P = (D == 128) ? 1 : (NT <= 5 ? 2 : 1);   // pages per warp step
  static constexpr int kTile = 16 * D * 2;                          // one page of K (or V)
  static constexpr int kStage = P * 2 * kTile;
  static constexpr int W = (D == 128 && P == 2) ? 6 : 8;            // warps per CTA
  static constexpr int kStages = (D == 128) ? (P == 2 ? 2 : 3) : (P == 2 ? 3 : 4);
  static constexpr size_t kStageBytes = size_t(W) * kStages * kStage;
  static constexpr size_t kSmem = kStageBytes + size_t(NT) * 8 * (2 * D + 16 + 4) +
                                  size_t(W) * kStages * 8 + 1024;
};

template <int D, int NT, bool CAPTURE>
__global__ void __launch_bounds__(VerifyCfg<D, NT>::W * 32, 1)
    verify_attn_kernel(const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap vmap, const VerifyParams p) {
  using Cfg = VerifyCfg<D, NT>;
  constexpr int W = Cfg::W;
  constexpr int P = Cfg::P;
  constexpr int NPAD = NT * 8;
  constexpr int STAGES = Cfg::kStages;
  constexpr int TILE = Cfg::kTile;
  constexpr int STAGE = Cfg::kStage;
  constexpr int QROW = 2 * D + 16;
  constexpr bool QS = Cfg::kQSmem;

  griddep_begin();

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* stage_area = smem;
  uint8_t* qs = smem + Cfg::kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(qs + NPAD * QROW);
  int* rawrow = reinterpret_cast<int*>(bars + W * STAGES);   // [NPAD] raw-logit row or -1

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int unit = b * p.hkv + g;
  const int T = p.gamma + 1;
  const int cap = p.max_pages * 16;
  int L = p.ctx_lens[b];
  if (L < 0 || L + T > cap) {
    if (tid == 0) set_error(p.err, kErrDeviceFault);
    L = max(0, min(L, cap - T));
  }
  const int npages = (L + T + 15) / 16;
  const int pbeg = split * p.pages_per_split;
  const int pend = min(pbeg + p.pages_per_split, npages);
  const int nsteps = pend > pbeg ? (pend - pbeg + P - 1) / P : 0;
  const int nmy = warp < nsteps ? (nsteps - warp + W - 1) / W : 0;
  // page pg of this warp's step i; a step past the split's end repeats its
  // first page (loaded, then masked) so every stage carries the same bytes
  auto step_page = [&](int i, int pg) {
    const int first = pbeg + P * (warp + i * W);
    return first + pg < pend ? first + pg : first;
  };

  if (tid == 0) {
    for (int i = 0; i < W * STAGES; ++i) mbar_init(smem_u32(&bars[i]), 1);
    fence_mbar_init();
  }
  const uint32_t stage0 = smem_u32(stage_area + warp * STAGES * STAGE);
  const uint32_t bar0 = smem_u32(&bars[warp * STAGES]);

  // Block-table entries of this warp's steps live in lane registers, 32 steps
  // per chunk, the next chunk loaded a chunk ahead.
  const int32_t* bt_row = p.block_table + size_t(b) * p.max_pages;
  int bt_cur[P], bt_nxt[P];
  auto bt_load = [&](int c, int (&dst)[P]) {
    const int i = c * 32 + lane;
#pragma unroll
    for (int pg = 0; pg < P; ++pg) dst[pg] = i < nmy ? __ldg(&bt_row[step_page(i, pg)]) : 0;
  };
  int bt_chunk = 0;
  bt_load(0, bt_cur);
  bt_load(1, bt_nxt);
  // Called by all lanes with increasing i; lane 0 issues the copies.
  auto issue = [&](int i) {
    const int c = i >> 5;
    if (c != bt_chunk) {
#pragma unroll
      for (int pg = 0; pg < P; ++pg) bt_cur[pg] = bt_nxt[pg];
      bt_load(c + 1, bt_nxt);
      bt_chunk = c;
    }
    int phys[P];
#pragma unroll
    for (int pg = 0; pg < P; ++pg) phys[pg] = __shfl_sync(0xffffffffu, bt_cur[pg], i & 31);
    if (lane == 0) {
      const int s = i % STAGES;
      const uint32_t bar = bar0 + s * 8;
      const uint32_t dst = stage0 + s * STAGE;
      mbar_arrive_expect_tx(bar, STAGE);
      // read once per pass: the tiles leave L2 first, so the scores, queries
      // and block table stay there for the kernels after this
      const uint64_t pol = l2_evict_first_policy();
#pragma unroll
      for (int pg = 0; pg < P; ++pg) {
        int ph = phys[pg];
        if (ph < 0 || ph >= p.num_pages) {
          set_error(p.err, kErrDeviceFault);
          ph = 0;
        }
        const int row = (ph * p.hkv + g) * 16;
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          tma_load_2d_hint(dst + pg * TILE + h * 2048, &kmap, h * 64, row, bar, pol);
          tma_load_2d_hint(dst + (P + pg) * TILE + h * 2048, &vmap, h * 64, row, bar, pol);
        }
      }
    }
  };

  // Q tile: column n = t * G + (h - g * G) for n < nq; with capture, columns
  // cap0 and cap0 + 1 (cap0 = nq rounded up to even) hold the summed captured
  // query, split into a bf16 part and a bf16 remainder; other columns are 0.
  const int cap0 = (p.nq + 1) & ~1;
  {
    constexpr int kChunks = NPAD * (D / 8);
    constexpr int kPer = (kChunks + W * 32 - 1) / (W * 32);
    uint4 v[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int i = tid + u * W * 32;
      const int n = i / (D / 8), c = i % (D / 8);
      v[u] = make_uint4(0, 0, 0, 0);
      if (i < kChunks && n < p.nq) {
        const int t = n / p.group, hl = n - t * p.group;
        v[u] = reinterpret_cast<const uint4*>(
            reinterpret_cast<const __nv_bfloat16*>(p.q) +
            ((size_t(b) * T + t) * p.hq + g * p.group + hl) * D)[c];
      }
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int i = tid + u * W * 32;
      if (i < kChunks)
        *reinterpret_cast<uint4*>(qs + (i / (D / 8)) * QROW + (i % (D / 8)) * 16) = v[u];
    }
  }
  if (CAPTURE) {
    __syncthreads();
    for (int j = tid; j < D; j += W * 32) {
      float acc = 0.f;
      for (int t = 0; t <= p.gamma; ++t) {
        if (!((p.row_mask >> t) & 1u)) continue;
        const __nv_bfloat16* src =
            reinterpret_cast<const __nv_bfloat16*>(p.q) + ((size_t(b) * T + t) * p.hq + g * p.group) * D;
        for (int hl = 0; hl < p.group; ++hl) acc += __bfloat162float(src[hl * D + j]);
      }
      const __nv_bfloat16 hi = __float2bfloat16_rn(acc);
      const __nv_bfloat16 lo = __float2bfloat16_rn(acc - __bfloat162float(hi));
      reinterpret_cast<__nv_bfloat16*>(qs + cap0 * QROW)[j] = hi;
      reinterpret_cast<__nv_bfloat16*>(qs + (cap0 + 1) * QROW)[j] = lo;
    }
  }
  __syncthreads();
  for (int i = 0; i < min(STAGES, nmy); ++i) issue(i);
  __syncwarp();

  uint32_t qf[QS ? 1 : D / 16][NT][2];
  if constexpr (!QS) load_q_frags<D, NT>(smem_u32(qs), qf);
  WarpState<D, NT> st;
  st.init();

  // Columns of this lane that enter the softmax: the real query rows only.
  uint32_t colbits = 0;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e)
      if (nt * 8 + 2 * (lane & 3) + e < p.nq) colbits |= 1u << (2 * nt + e);
  const bool cap_lane = CAPTURE && (lane & 3) == ((cap0 & 7) >> 1);
  const int cap_nt = cap0 >> 3;
  float* srow = CAPTURE ? p.scores + size_t(unit) * p.score_stride : nullptr;
  int Lcap = L;   // captured positions [0, L), written only inside the score row
  if (CAPTURE && L > p.score_stride) {
    if (tid == 0) set_error(p.err, kErrDeviceFault);
    Lcap = p.score_stride;
  }
  const int last_valid = L + p.gamma;
  // raw-logit mode: column n = t * G + hl of a captured row t goes to row
  // (b * R + rank of t among the captured rows) * Hq + g * G + hl
  const bool raw = !CAPTURE && p.raw != nullptr;
  if (raw) {
    for (int n = tid; n < NPAD; n += W * 32) {
      int rr = -1;
      if (n < p.nq) {
        const int t = n / p.group, hl = n - t * p.group;
        if ((p.row_mask >> t) & 1u)
          rr = (b * p.raw_rows + __popc(p.row_mask & ((1u << t) - 1u))) * p.hq + g * p.group + hl;
      }
      rawrow[n] = rr;
    }
    __syncthreads();
  }
  const int Lraw = raw ? min(L, p.raw_stride) : 0;

  int done = 0;
  bool ok = true;
  for (; done < nmy; ++done) {
    const int i = done;
    const int s = i % STAGES;
    if (!mbar_wait_bounded(bar0 + s * 8, (i / STAGES) & 1)) {
      ok = false;
      break;
    }
    uint32_t kb[P], vb[P];
    int pos0[P];
    bool live[P];
#pragma unroll
    for (int pg = 0; pg < P; ++pg) {
      const int first = pbeg + P * (warp + i * W);
      live[pg] = first + pg < pend;
      pos0[pg] = step_page(i, pg) * 16;
      kb[pg] = stage0 + s * STAGE + pg * TILE;
      vb[pg] = stage0 + s * STAGE + (P + pg) * TILE;
      if (pos0[pg] + 15 > last_valid) {
        // Slots past the window hold whatever the cache holds there; zero
        // their V rows so that a 0 probability never meets a NaN.
        uint8_t* vgen = stage_area + (warp * STAGES + s) * STAGE + (P + pg) * TILE;
        const int first_bad = last_valid + 1 - pos0[pg];
        for (int j = lane; j < (16 - first_bad) * (D / 8); j += 32) {
          const int r = first_bad + j / (D / 8), c = j % (D / 8);
          *reinterpret_cast<uint4*>(vgen + SwizzledTile::addr(0, r, c)) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
    }
    float sc[P][NT][4];
    if constexpr (QS)
      tile_scores_qsmem<D, NT, P, SwizzledTile>(kb, smem_u32(qs), sc);
    else
      tile_scores<D, NT, P, SwizzledTile>(kb, qf, sc);
    if (cap_lane) {
#pragma unroll
      for (int pg = 0; pg < P; ++pg) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          if (nt == cap_nt && live[pg]) {
            const int pa = pos0[pg] + (lane >> 2);
            if (pa < Lcap) srow[pa] = (sc[pg][nt][0] + sc[pg][nt][1]) * p.scale;
            if (pa + 8 < Lcap) srow[pa + 8] = (sc[pg][nt][2] + sc[pg][nt][3]) * p.scale;
          }
      }
    }
    if (raw) {
      // the pages' way: every captured row's logit of every head goes to memory
#pragma unroll
      for (int pg = 0; pg < P; ++pg)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int n = nt * 8 + 2 * (lane & 3) + (k & 1);
            const int pos = pos0[pg] + (lane >> 2) + 8 * (k >> 1);
            const int rr = rawrow[n];
            if (live[pg] && rr >= 0 && pos < Lraw)
              p.raw[size_t(rr) * p.raw_stride + pos] = sc[pg][nt][k] * p.scale;
          }
    }
    float x[P][NT][4];
#pragma unroll
    for (int pg = 0; pg < P; ++pg) {
      const bool need_mask = pos0[pg] + 15 > L;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float v = sc[pg][nt][k] * p.scale_log2;
          if (!live[pg] || !((colbits >> (2 * nt + (k & 1))) & 1u)) v = -INFINITY;
          if (need_mask) {
            const int pos = pos0[pg] + (lane >> 2) + 8 * (k >> 1);
            const int n = nt * 8 + 2 * (lane & 3) + (k & 1);
            const int t = min(n / p.group, p.gamma);
            if (pos > L + t) v = -INFINITY;
          }
          x[pg][nt][k] = v;
        }
    }
    tile_softmax_pv<D, NT, P, SwizzledTile>(st, x, vb);
    __syncwarp();
    if (i + STAGES < nmy) {
      fence_proxy_async_smem();
      issue(i + STAGES);
    }
  }
  if (!ok) {
    if (lane == 0) set_error(p.err, kErrDeviceTimeout);
    // Let the copies already issued land before the CTA's shared memory is reused.
    for (int j = done; j < min(done + STAGES, nmy); ++j)
      (void)mbar_wait_bounded(bar0 + (j % STAGES) * 8, (j / STAGES) & 1);
  }
  reduce_row_sums<D, NT>(st);
  __syncthreads();

  SplitWorkspace ws{p.tickets, p.part_ml, p.part_o};
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
  auto out_row = [&](int n) {
    const int t = n / p.group, hl = n - t * p.group;
    return out + ((size_t(b) * T + t) * p.hq + g * p.group + hl) * D;
  };
  merge_and_write<D, NT, W>(st, stage_area, Cfg::kStageBytes, p.nq, unit, split, p.num_splits, ws,
                            out_row);
}

#if defined(VEGAS_D) && defined(VEGAS_CAP)
// This translation unit instantiates the kernels of one (head_dim, capture)
// pair; the build compiles it once per pair so the units compile in parallel.
template <int D, int NT, bool CAP>
static cudaError_t launch_one(const CUtensorMap& kmap, const CUtensorMap& vmap,
                              const VerifyParams& p, int batch, cudaStream_t stream) {
  using Cfg = VerifyCfg<D, NT>;
  static std::atomic<uint32_t> configured{0};
  cudaError_t e = once_per_device(configured, [] {
    return cudaFuncSetAttribute(verify_attn_kernel<D, NT, CAP>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::kSmem);
  });
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.num_splits, p.hkv, batch);
  cfg.blockDim = dim3(Cfg::W * 32, 1, 1);
  cfg.dynamicSmemBytes = Cfg::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, verify_attn_kernel<D, NT, CAP>, kmap, vmap, p);
}

template <>
cudaError_t launch_verify_t<VEGAS_D, (VEGAS_CAP != 0)>(const CUtensorMap& kmap,
                                                       const CUtensorMap& vmap,
                                                       const VerifyParams& p, int ntiles,
                                                       int batch, cudaStream_t s) {
  constexpr int D = VEGAS_D;
  constexpr bool CAP = VEGAS_CAP != 0;
  switch (ntiles) {
    case 1: return launch_one<D, 1, CAP>(kmap, vmap, p, batch, s);
    case 2: return launch_one<D, 2, CAP>(kmap, vmap, p, batch, s);
    case 3: return launch_one<D, 3, CAP>(kmap, vmap, p, batch, s);
    case 4: return launch_one<D, 4, CAP>(kmap, vmap, p, batch, s);
    case 5: return launch_one<D, 5, CAP>(kmap, vmap, p, batch, s);
    case 6: return launch_one<D, 6, CAP>(kmap, vmap, p, batch, s);
#if VEGAS_D == 64
    case 7: return launch_one<D, 7, CAP>(kmap, vmap, p, batch, s);
    case 8: return launch_one<D, 8, CAP>(kmap, vmap, p, batch, s);
#endif
    default: return cudaErrorInvalidValue;
  }
}
#endif

}  // namespace vegas
