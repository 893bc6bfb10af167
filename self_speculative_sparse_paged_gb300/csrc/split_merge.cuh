// Merging partial softmax states into the attention output.
//
// Stage 1 (inside a CTA): the W warps' (m, l, O^T) states are merged in shared
// memory.  Stage 2 (across the S CTAs of one (sequence, KV head) unit): each
// CTA writes its merged partial to the workspace, bumps the unit's ticket, and
// the CTA that arrives last merges all S partials and writes bf16 output.  No
// CTA waits for another; the last one resets the ticket to zero.
//
// Merge rule (flash-decoding): M = max_s m_s, f_s = 2^(m_s - M), l = sum_s
// f_s l_s, O = sum_s f_s O_s / l (a part that attended nothing has l_s = 0).
#pragma once

#include "attn_core.cuh"

namespace vegas {

struct SplitWorkspace {
  int* tickets;     // [units]
  float* part_ml;   // [units][S][nq][2]: (m, l)
  float* part_o;    // [units][S][nq][D]
};

// After every thread of the CTA has written this CTA's partial states (m, l,
// O): takes the unit's ticket and, in the last of the unit's num_ctas CTAs to
// arrive, merges the unit's num_splits partials (one or more per CTA) into
// bf16 output rows.  Called by all NTH threads of the CTA; `area` is free
// shared memory of at least 3 * num_splits * nq floats, `flag` one int of
// shared memory.
template <int D, int NTH, int NQMAX, class OutRow>
__device__ __forceinline__ void finish_splits(const SplitWorkspace& ws, int unit, int num_ctas,
                                              int num_splits, int nq, OutRow out_row,
                                              float* area, int* flag) {
  constexpr int E = (NQMAX * D + NTH - 1) / NTH;   // elements per thread, nq <= NQMAX
  const int tid = threadIdx.x;
  const int nel = nq * D;
  __threadfence();
  __syncthreads();
  if (tid == 0) *flag = (atomicAdd(&ws.tickets[unit], 1) == num_ctas - 1);
  __syncthreads();
  if (!*flag) return;
  __threadfence();

  // Every split's (m, l) is staged in shared memory by one parallel sweep and
  // turned into weights w[s][n] = f_s / l; the partial outputs are then summed
  // with loads issued in independent batches.
  float* wS = area;                        // [num_splits][nq]
  float* mS = wS + num_splits * nq;        // [num_splits][nq]
  float* lS = mS + num_splits * nq;        // [num_splits][nq]
  const size_t base = (size_t)unit * num_splits;
  const float2* ml = reinterpret_cast<const float2*>(ws.part_ml) + base * nq;
  for (int i = tid; i < num_splits * nq; i += NTH) {
    const float2 v = __ldcg(&ml[i]);
    mS[i] = v.x;
    lS[i] = v.y;
  }
  __syncthreads();
  for (int n = tid; n < nq; n += NTH) {
    float M = -INFINITY;
    for (int s = 0; s < num_splits; ++s) M = fmaxf(M, mS[s * nq + n]);
    float L = 0.f;
    for (int s = 0; s < num_splits; ++s) {
      const float ms = mS[s * nq + n];
      const float f = (ms == -INFINITY) ? 0.f : ex2(ms - M);
      wS[s * nq + n] = f;
      L += f * lS[s * nq + n];
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    for (int s = 0; s < num_splits; ++s) wS[s * nq + n] *= inv;
  }
  __syncthreads();
  // Every split wrote a partial O (zeros where it attended nothing), so the
  // weighted sum needs no branch.  Element e = n * D + dim of split s sits at
  // part_o[(base + s) * nq * D + e]; a thread owns E4 groups of 4 consecutive
  // elements and keeps U splits' loads in flight at once.
  (void)E;
  constexpr int E4 = (NQMAX * D / 4 + NTH - 1) / NTH;
  constexpr int U = 8;
  const int nel4 = nel / 4;
  const float4* po = reinterpret_cast<const float4*>(ws.part_o + base * nq * D);
  float4 a[E4];
#pragma unroll
  for (int j = 0; j < E4; ++j) a[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < num_splits; s0 += U) {
    float4 v[U][E4];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int j = 0; j < E4; ++j) {
        const int e4 = tid + j * NTH;
        v[u][j] = (s0 + u < num_splits && e4 < nel4) ? __ldcg(&po[size_t(s0 + u) * nel4 + e4])
                                                      : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int j = 0; j < E4; ++j) {
        const int n = min((tid + j * NTH) * 4 / D, nq - 1);
        const float w = s0 + u < num_splits ? wS[(s0 + u) * nq + n] : 0.f;
        a[j].x += w * v[u][j].x;
        a[j].y += w * v[u][j].y;
        a[j].z += w * v[u][j].z;
        a[j].w += w * v[u][j].w;
      }
  }
#pragma unroll
  for (int j = 0; j < E4; ++j) {
    const int e4 = tid + j * NTH;
    if (e4 < nel4) {
      const int e = e4 * 4;
      __nv_bfloat16* dst = out_row(e / D) + e % D;
      *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(a[j].x, a[j].y);
      *reinterpret_cast<__nv_bfloat162*>(dst + 2) = __floats2bfloat162_rn(a[j].z, a[j].w);
    }
  }
  if (tid == 0) ws.tickets[unit] = 0;
}

// Merges the W warps' states of a CTA into shared memory: outM[n], outL[n]
// (running max and row sum of column n) and outO[n * D + dim] (unnormalised
// output), for n < nq.  Called by every thread after reduce_row_sums; `area`
// is free shared memory of `area_bytes` (the drained stage buffers), distinct
// from the out arrays.
template <int D, int NT, int W>
__device__ __forceinline__ void cta_merge_to_smem(const WarpState<D, NT>& st, uint8_t* area,
                                                  size_t area_bytes, int nq, float* outM,
                                                  float* outL, float* outO) {
  constexpr int NPAD = NT * 8;
  constexpr int OS = D + 4;
  constexpr int NTH = W * 32;
  constexpr int E = (NPAD * D + NTH - 1) / NTH;
  const int nel = nq * D;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  float* cm = reinterpret_cast<float*>(area);          // [W][NPAD] -> becomes f_w
  float* cl = cm + W * NPAD;                           // [W][NPAD]
  float* cO = reinterpret_cast<float*>(area + 4096 * ((2 * W * NPAD * 4 + 4095) / 4096));
  const size_t o_bytes = area_bytes - (reinterpret_cast<uint8_t*>(cO) - area);
  const int C = min(W, (int)(o_bytes / (size_t(NPAD) * OS * 4)));
  if ((lane >> 2) == 0) {
    const int c = 2 * (lane & 3);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        cm[warp * NPAD + nt * 8 + c + e] = st.m[nt][e];
        cl[warp * NPAD + nt * 8 + c + e] = st.l[nt][e];
      }
  }
  __syncthreads();
  for (int n = tid; n < NPAD; n += NTH) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < W; ++w) M = fmaxf(M, cm[w * NPAD + n]);
    float lsum = 0.f;
#pragma unroll
    for (int w = 0; w < W; ++w) {
      const float f = ex2(cm[w * NPAD + n] - M);
      cm[w * NPAD + n] = f;
      lsum += f * cl[w * NPAD + n];
    }
    if (n < nq) {
      outM[n] = M;
      outL[n] = lsum;
    }
  }
  float acc[E];
#pragma unroll
  for (int j = 0; j < E; ++j) acc[j] = 0.f;
  for (int w0 = 0; w0 < W; w0 += C) {
    if (warp >= w0 && warp < w0 + C) stage_warp_o<D, NT>(st, cO, warp - w0);
    __syncthreads();
#pragma unroll
    for (int j = 0; j < E; ++j) {
      const int e = tid + j * NTH;
      const int n = e / D, dim = e % D;
      if (e < nel)
        for (int w = w0; w < min(W, w0 + C); ++w)
          acc[j] += cm[w * NPAD + n] * cO[((w - w0) * NPAD + n) * OS + dim];
    }
    __syncthreads();
  }
#pragma unroll
  for (int j = 0; j < E; ++j) {
    const int e = tid + j * NTH;
    if (e < nel) outO[e] = acc[j];
  }
}

// Called by every thread of the CTA after the main loop, with row sums already
// reduced (reduce_row_sums).  `area` is free shared memory of `area_bytes`
// (the drained stage buffers).  out_row(n) returns the bf16 output row of
// query column n < nq.
template <int D, int NT, int W, class OutRow>
__device__ __forceinline__ void merge_and_write(const WarpState<D, NT>& st, uint8_t* area,
                                                size_t area_bytes, int nq, int unit, int split,
                                                int num_splits, const SplitWorkspace& ws,
                                                OutRow out_row) {
  constexpr int NPAD = NT * 8;
  constexpr int OS = D + 4;
  constexpr int NTH = W * 32;
  constexpr int E = (NPAD * D + NTH - 1) / NTH;   // output elements owned per thread
  const int nel = nq * D;                          // element e = n * D + dim, n < nq
  const int tid = threadIdx.x;
  const int warp = tid >> 5;

  float* cm = reinterpret_cast<float*>(area);          // [W][NPAD] -> becomes f_w
  float* cl = cm + W * NPAD;                           // [W][NPAD]
  float* colM = cl + W * NPAD;                         // [NPAD]
  float* colL = colM + NPAD;                           // [NPAD]
  int* flag = reinterpret_cast<int*>(colL + NPAD);
  float* cO = reinterpret_cast<float*>(area + 4096 * ((2 * W * NPAD * 4 + 2 * NPAD * 4 + 16 + 4095) / 4096));
  const size_t o_bytes = area_bytes - (reinterpret_cast<uint8_t*>(cO) - area);
  const int C = min(W, (int)(o_bytes / (size_t(NPAD) * OS * 4)));   // warps staged per round

  // per-warp (m, l)
  {
    const int lane = tid & 31;
    if ((lane >> 2) == 0) {
      const int c = 2 * (lane & 3);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          cm[warp * NPAD + nt * 8 + c + e] = st.m[nt][e];
          cl[warp * NPAD + nt * 8 + c + e] = st.l[nt][e];
        }
    }
  }
  __syncthreads();
  for (int n = tid; n < NPAD; n += NTH) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < W; ++w) M = fmaxf(M, cm[w * NPAD + n]);
    float lsum = 0.f;
#pragma unroll
    for (int w = 0; w < W; ++w) {
      const float mw = cm[w * NPAD + n];
      const float f = (mw == -INFINITY) ? 0.f : ex2(mw - M);
      cm[w * NPAD + n] = f;
      lsum += f * cl[w * NPAD + n];
    }
    colM[n] = M;
    colL[n] = lsum;
  }
  float acc[E];
#pragma unroll
  for (int j = 0; j < E; ++j) acc[j] = 0.f;
  for (int w0 = 0; w0 < W; w0 += C) {
    if (warp >= w0 && warp < w0 + C) stage_warp_o<D, NT>(st, cO, warp - w0);
    __syncthreads();
#pragma unroll
    for (int j = 0; j < E; ++j) {
      const int e = tid + j * NTH;
      const int n = e / D, dim = e % D;
      if (e < nel)
        for (int w = w0; w < min(W, w0 + C); ++w)
          acc[j] += cm[w * NPAD + n] * cO[((w - w0) * NPAD + n) * OS + dim];
    }
    __syncthreads();
  }

  if (num_splits == 1) {
#pragma unroll
    for (int j = 0; j < E; ++j) {
      const int e = tid + j * NTH;
      const int n = e / D, dim = e % D;
      if (n < nq) {
        const float L = colL[n];
        out_row(n)[dim] = __float2bfloat16_rn(L > 0.f ? acc[j] / L : 0.f);
      }
    }
    return;
  }

  const size_t part = (size_t)unit * num_splits + split;
#pragma unroll
  for (int j = 0; j < E; ++j) {
    const int e = tid + j * NTH;
    const int n = e / D, dim = e % D;
    if (n < nq) {
      ws.part_o[(part * nq + n) * D + dim] = acc[j];
      if (dim == 0) {
        ws.part_ml[(part * nq + n) * 2 + 0] = colM[n];
        ws.part_ml[(part * nq + n) * 2 + 1] = colL[n];
      }
    }
  }
  finish_splits<D, NTH, NPAD>(ws, unit, num_splits, num_splits, nq, out_row, cO, flag);
}

}  // namespace vegas
