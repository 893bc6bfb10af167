// Merging partial softmax states into the attention output.
//
// Stage 1 (inside a CTA): the W warps' (m, l, O^T) states are merged in shared
// memory.  Stage 2 (across the S CTAs of one (sequence, KV head) unit): each
// CTA writes its merged partial to the workspace, bumps the unit's ticket, and
// the CTA that arrives last merges all S partials and writes bf16 output.  No
// CTA waits for another; the last one resets the ticket to zero.
//
// Merge rule (flash-decoding): M = max_s m_s, f_s = 2^(m_s - M) (0 when
// m_s = -inf), l = sum_s f_s l_s, O = sum_s f_s O_s / l.
#pragma once

#include "attn_core.cuh"

namespace vegas {

struct SplitWorkspace {
  int* tickets;     // [units]
  float* part_ml;   // [units][S][nq][2]: (m, l)
  float* part_o;    // [units][S][nq][D]
};

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
  __threadfence();
  __syncthreads();
  if (tid == 0) *flag = (atomicAdd(&ws.tickets[unit], 1) == num_splits - 1);
  __syncthreads();
  if (!*flag) return;
  __threadfence();

  // Last CTA of the unit.  Every split's (m, l) is staged in shared memory by
  // one parallel sweep and turned into weights w[s][n] = f_s / l; the partial
  // outputs are then summed with loads issued in independent batches.
  float* wS = cO;                          // [num_splits][nq]
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
  // part_o[(base + s) * nq * D + e].
  const float* po = ws.part_o + base * nq * D;
  float a[E];
#pragma unroll
  for (int j = 0; j < E; ++j) a[j] = 0.f;
  constexpr int U = 4;
  int s = 0;
  for (; s + U <= num_splits; s += U) {
    float v[U][E];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int j = 0; j < E; ++j) {
        const int e = tid + j * NTH;
        v[u][j] = e < nel ? __ldcg(&po[size_t(s + u) * nel + e]) : 0.f;
      }
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int j = 0; j < E; ++j) {
        const int n = min((tid + j * NTH) / D, nq - 1);
        a[j] += wS[(s + u) * nq + n] * v[u][j];
      }
  }
  for (; s < num_splits; ++s) {
#pragma unroll
    for (int j = 0; j < E; ++j) {
      const int e = tid + j * NTH;
      if (e < nel) a[j] += wS[s * nq + e / D] * __ldcg(&po[size_t(s) * nel + e]);
    }
  }
#pragma unroll
  for (int j = 0; j < E; ++j) {
    const int e = tid + j * NTH;
    if (e < nel) out_row(e / D)[e % D] = __float2bfloat16_rn(a[j]);
  }
  if (tid == 0) ws.tickets[unit] = 0;
}

}  // namespace vegas
