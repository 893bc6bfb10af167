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
// sequence).  Each of the 8 warps walks its own pages of the split (page
// w, w+8, ...) through a private ring of TMA stages: one 16-token page of K and
// of V per stage, loaded with 2-D tensor TMA (128-byte swizzle) straight from
// the paged cache, one mbarrier per stage.  The warp computes S^T for all
// (gamma+1)*G query rows of the unit at once (positions x query rows), adds
// the captured rows' logits per position and writes the fp32 score, then runs
// the lazy online softmax and O^T += V^T P^T.  Warp states merge in shared
// memory, splits merge through the workspace (last-arriving CTA).
#include "kernels.h"
#include "split_merge.cuh"

namespace vegas {

template <int D>
struct VerifyCfg {
  static constexpr int kStages = (D == 128) ? 3 : 4;
  static constexpr int kTile = 16 * D * 2;      // one page of K (or V) for one KV head
  static constexpr int kStage = 2 * kTile;
  static constexpr int kMaxNT = (D == 128) ? 6 : 8;
  __host__ __device__ static constexpr bool q_in_smem(int nt) {
    return (D == 128) ? nt >= 4 : nt >= 7;
  }
};

template <int D, int NT>
constexpr size_t verify_smem_layout_bytes() {
  return size_t(kAttnWarps) * VerifyCfg<D>::kStages * VerifyCfg<D>::kStage   // stages
         + size_t(NT) * 8 * (2 * D + 16)                                     // Q tile
         + size_t(kAttnWarps) * VerifyCfg<D>::kStages * 8                    // mbarriers
         + 1024;                                                             // alignment slack
}

template <int D, int NT, bool CAPTURE>
__global__ void __launch_bounds__(kAttnWarps * 32, 1)
    verify_attn_kernel(const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap vmap, const VerifyParams p) {
  constexpr int W = kAttnWarps;
  constexpr int NPAD = NT * 8;
  constexpr int STAGES = VerifyCfg<D>::kStages;
  constexpr int TILE = VerifyCfg<D>::kTile;
  constexpr int STAGE = VerifyCfg<D>::kStage;
  constexpr int QROW = 2 * D + 16;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* stage_area = smem;
  uint8_t* qs = smem + W * STAGES * STAGE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(qs + NPAD * QROW);

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

  if (tid == 0) {
    for (int i = 0; i < W * STAGES; ++i) mbar_init(smem_u32(&bars[i]), 1);
    fence_mbar_init();
  }
  // Q rows of the unit, column n = t * G + (h - g * G); rows past nq are zero.
  for (int i = tid; i < NPAD * (D / 8); i += W * 32) {
    const int n = i / (D / 8), c = i % (D / 8);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (n < p.nq) {
      const int t = n / p.group, hl = n - t * p.group;
      const uint4* src = reinterpret_cast<const uint4*>(
          reinterpret_cast<const __nv_bfloat16*>(p.q) +
          ((size_t(b) * T + t) * p.hq + g * p.group + hl) * D);
      v = src[c];
    }
    *reinterpret_cast<uint4*>(qs + n * QROW + c * 16) = v;
  }
  __syncthreads();

  const int first = pbeg + warp;
  const int nmy = first < pend ? (pend - first + W - 1) / W : 0;
  const uint32_t stage0 = smem_u32(stage_area + warp * STAGES * STAGE);
  const uint32_t bar0 = smem_u32(&bars[warp * STAGES]);

  auto issue = [&](int i) {
    const int pg = first + i * W;
    const int s = i % STAGES;
    int phys = p.block_table[size_t(b) * p.max_pages + pg];
    if (phys < 0 || phys >= p.num_pages) {
      set_error(p.err, kErrDeviceFault);
      phys = 0;
    }
    const int row = (phys * p.hkv + g) * 16;
    const uint32_t bar = bar0 + s * 8;
    const uint32_t kdst = stage0 + s * STAGE;
    mbar_arrive_expect_tx(bar, STAGE);
#pragma unroll
    for (int h = 0; h < D / 64; ++h) {
      tma_load_2d(kdst + h * 2048, &kmap, h * 64, row, bar);
      tma_load_2d(kdst + TILE + h * 2048, &vmap, h * 64, row, bar);
    }
  };
  if (lane == 0) {
    for (int i = 0; i < min(STAGES, nmy); ++i) issue(i);
  }
  __syncwarp();

  // Q^T fragments live in registers unless the O^T accumulator leaves no room.
  constexpr bool QS = VerifyCfg<D>::q_in_smem(NT);
  uint32_t qf[QS ? 1 : D / 16][NT][2];
  if constexpr (!QS) load_q_frags<D, NT>(smem_u32(qs), qf);
  WarpState<D, NT> st;
  st.init();

  uint32_t capbits = 0;
  if (CAPTURE) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int n = nt * 8 + 2 * (lane & 3) + e;
        if (n < p.nq) {
          const int t = n / p.group;
          if (t == p.row_a || t == p.row_b) capbits |= 1u << (2 * nt + e);
        }
      }
  }
  float* srow = CAPTURE ? p.scores + size_t(unit) * p.score_stride : nullptr;
  int Lcap = L;   // captured positions: [0, L), written only inside the score row
  if (CAPTURE && L > p.score_stride) {
    if (tid == 0) set_error(p.err, kErrDeviceFault);
    Lcap = p.score_stride;
  }
  const int last_valid = L + p.gamma;

  int done = 0;
  bool ok = true;
  for (; done < nmy; ++done) {
    const int i = done;
    const int s = i % STAGES;
    if (!mbar_wait_bounded(bar0 + s * 8, (i / STAGES) & 1)) {
      ok = false;
      break;
    }
    const int pos0 = (first + i * W) * 16;
    const uint32_t kb = stage0 + s * STAGE;
    const uint32_t vb = kb + TILE;
    if (pos0 + 15 > last_valid) {
      // Slots past the window hold whatever the cache holds there; zero their
      // V rows so that a 0 probability never meets a NaN.
      uint8_t* vgen = stage_area + (warp * STAGES + s) * STAGE + TILE;
      const int first_bad = last_valid + 1 - pos0;
      for (int j = lane; j < (16 - first_bad) * (D / 8); j += 32) {
        const int r = first_bad + j / (D / 8), c = j % (D / 8);
        *reinterpret_cast<uint4*>(vgen + SwizzledTile::addr(0, r, c)) = make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();
      __syncwarp();
    }
    float sc[NT][4];
    if constexpr (QS)
      tile_scores_qsmem<D, NT, SwizzledTile>(kb, smem_u32(qs), sc);
    else
      tile_scores<D, NT, SwizzledTile>(kb, qf, sc);
    if (CAPTURE && pos0 < L) {
      float c0 = 0.f, c1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e)
          if ((capbits >> (2 * nt + e)) & 1u) {
            c0 += sc[nt][e];
            c1 += sc[nt][2 + e];
          }
      c0 += __shfl_xor_sync(0xffffffffu, c0, 1);
      c0 += __shfl_xor_sync(0xffffffffu, c0, 2);
      c1 += __shfl_xor_sync(0xffffffffu, c1, 1);
      c1 += __shfl_xor_sync(0xffffffffu, c1, 2);
      if ((lane & 3) == 0) {
        const int pa = pos0 + (lane >> 2);
        if (pa < Lcap) srow[pa] = c0 * p.scale;
        if (pa + 8 < Lcap) srow[pa + 8] = c1 * p.scale;
      }
    }
    float x[NT][4];
    const bool need_mask = pos0 + 15 > L;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float v = sc[nt][k] * p.scale_log2;
        if (need_mask) {
          const int pos = pos0 + (lane >> 2) + 8 * (k >> 1);
          const int n = nt * 8 + 2 * (lane & 3) + (k & 1);
          const int t = min(n / p.group, p.gamma);
          if (pos > L + t) v = -INFINITY;
        }
        x[nt][k] = v;
      }
    tile_softmax_pv<D, NT, SwizzledTile>(st, x, vb);
    __syncwarp();
    if (i + STAGES < nmy && lane == 0) {
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
  merge_and_write<D, NT, W>(st, stage_area, size_t(W) * STAGES * STAGE, p.nq, unit, split,
                            p.num_splits, ws, out_row);
}

static size_t verify_smem_bytes(int head_dim, int ntiles) {
  (void)ntiles;  // sized for the largest tile count so one attribute fits every launch
  return head_dim == 128 ? verify_smem_layout_bytes<128, VerifyCfg<128>::kMaxNT>()
                         : verify_smem_layout_bytes<64, VerifyCfg<64>::kMaxNT>();
}

#if defined(VEGAS_D) && defined(VEGAS_CAP)
// This translation unit instantiates the kernels of one (head_dim, capture)
// pair; the build compiles it once per pair so the units compile in parallel.
template <int D, int NT, bool CAP>
static cudaError_t launch_one(const CUtensorMap& kmap, const CUtensorMap& vmap,
                              const VerifyParams& p, int batch, cudaStream_t stream) {
  const size_t smem = verify_smem_bytes(D, NT);
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(verify_attn_kernel<D, NT, CAP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid(p.num_splits, p.hkv, batch);
  verify_attn_kernel<D, NT, CAP><<<grid, kAttnWarps * 32, smem, stream>>>(kmap, vmap, p);
  return cudaGetLastError();
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
