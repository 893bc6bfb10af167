// Warp-level attention over 16-position tiles, shared by the verify and the
// sparse draft kernels.
//
// Orientation: positions are the MMA's M dimension and query rows its N
// dimension.  One warp computes S^T = K_tile (16 x D) * Q^T (D x 8*NT) with
// mma.sync m16n8k16 (bf16 in, fp32 accumulate), so the (gamma+1)*G query rows
// of a (sequence, KV head) pad only to a multiple of 8.  The probabilities
// P^T are turned into the B operand of O^T += V^T (D x 16) * P^T (16 x 8*NT)
// by one movmatrix transpose per 8x8 block, without touching shared memory.
//
// Fragment ownership (lane l, r = l / 4, c = 2 * (l % 4)):
//   S tile  s[nt][0..3]: positions (r, r, r+8, r+8), query columns
//                        (8nt+c, 8nt+c+1, 8nt+c, 8nt+c+1)
//   O^T     o[mt][nt][0..3]: dims (16mt+r, 16mt+r, 16mt+r+8, 16mt+r+8), same columns
//   m[nt][e], l[nt][e]: running max (log2 units) / partial sum of column 8nt+c+e
//
// Softmax: logits are kept in log2 units (x = s * scale * log2 e).  The
// running max is raised only when some logit exceeds it by more than
// kRescaleSlack, decided by one warp vote per tile; otherwise probabilities
// 2^(x - m) <= 2^kRescaleSlack are used directly (bf16/fp32 hold them
// exactly in range), which removes the per-tile max reduction.
#pragma once

#include "vegas_common.cuh"

namespace vegas {

constexpr float kRescaleSlack = 8.0f;
// Running max of a column that has seen no logit yet (finite, so that
// 2^(x - m) and 2^(m_old - m_new) never form inf - inf).
constexpr float kEmptyMax = -1.0e30f;
constexpr float kLog2e = 1.4426950408889634f;

// 16-row tile written by a 2-D TMA load with 128-byte swizzle: D/64 boxes of
// 16 rows x 128 bytes; the 16-byte chunk cc of row r sits at cc ^ (r % 8).
struct SwizzledTile {
  __device__ __forceinline__ static uint32_t addr(uint32_t base, int row, int chunk) {
    return base + (chunk >> 3) * 2048 + row * 128 + (((chunk & 7) ^ (row & 7)) << 4);
  }
};

// 16-row tile of plain rows at a padded stride (D*2 + 16 bytes), filled by
// per-row bulk copies; the pad makes 8-row ldmatrix reads conflict-free.
template <int D>
struct PaddedTile {
  static constexpr int kRowBytes = D * 2 + 16;
  __device__ __forceinline__ static uint32_t addr(uint32_t base, int row, int chunk) {
    return base + row * kRowBytes + chunk * 16;
  }
};

template <int D, int NT>
struct WarpState {
  float o[D / 16][NT][4];
  float m[NT][2];
  float l[NT][2];

  __device__ __forceinline__ void init() {
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) o[mt][nt][i] = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        m[nt][e] = kEmptyMax;
        l[nt][e] = 0.f;
      }
  }
};

// Q^T B-fragments for every (k-step, n-tile), from a padded Q tile in shared
// memory ([8*NT rows][D], row stride D*2 + 16 bytes).
template <int D, int NT>
__device__ __forceinline__ void load_q_frags(uint32_t q_base, uint32_t (&qf)[D / 16][NT][2]) {
  const int lane = threadIdx.x & 31;
  constexpr int kRow = D * 2 + 16;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int ks = 0; ks < D / 16; ks += 2) {
      const int row = nt * 8 + (lane & 7);
      const int chunk = 2 * ks + (lane >> 3);
      ldmatrix_x4(q_base + row * kRow + chunk * 16, qf[ks][nt][0], qf[ks][nt][1],
                  qf[ks + 1][nt][0], qf[ks + 1][nt][1]);
    }
}

// S^T for P 16-position tiles (one per page), the pages' MMA chains interleaved.
template <int D, int NT, int P, class Tile>
__device__ __forceinline__ void tile_scores(const uint32_t (&k_base)[P],
                                            const uint32_t (&qf)[D / 16][NT][2],
                                            float (&s)[P][NT][4]) {
  const int lane = threadIdx.x & 31;
  const int mi = lane >> 3;
  const int row = (lane & 7) + 8 * (mi & 1);
#pragma unroll
  for (int pg = 0; pg < P; ++pg)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) s[pg][nt][i] = 0.f;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    uint32_t a[P][4];
#pragma unroll
    for (int pg = 0; pg < P; ++pg)
      ldmatrix_x4(Tile::addr(k_base[pg], row, 2 * ks + (mi >> 1)), a[pg][0], a[pg][1], a[pg][2],
                  a[pg][3]);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int pg = 0; pg < P; ++pg)
        mma_bf16_16816(s[pg][nt], a[pg][0], a[pg][1], a[pg][2], a[pg][3], qf[ks][nt][0],
                       qf[ks][nt][1]);
  }
}

// As tile_scores, reading the Q^T fragments from the padded Q tile in shared
// memory at every k-step (used where registers are short).
template <int D, int NT, int P, class Tile>
__device__ __forceinline__ void tile_scores_qsmem(const uint32_t (&k_base)[P], uint32_t q_base,
                                                  float (&s)[P][NT][4]) {
  const int lane = threadIdx.x & 31;
  const int mi = lane >> 3;
  const int row = (lane & 7) + 8 * (mi & 1);
  constexpr int kRow = D * 2 + 16;
#pragma unroll
  for (int pg = 0; pg < P; ++pg)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) s[pg][nt][i] = 0.f;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    uint32_t a[P][4];
#pragma unroll
    for (int pg = 0; pg < P; ++pg)
      ldmatrix_x4(Tile::addr(k_base[pg], row, 2 * ks + (mi >> 1)), a[pg][0], a[pg][1], a[pg][2],
                  a[pg][3]);
#pragma unroll
    for (int nt = 0; nt < NT; nt += 2) {
      if (nt + 1 < NT) {
        uint32_t b0, b1, b2, b3;
        const int qrow = (nt + (mi >> 1)) * 8 + (lane & 7);
        ldmatrix_x4(q_base + qrow * kRow + (2 * ks + (mi & 1)) * 16, b0, b1, b2, b3);
#pragma unroll
        for (int pg = 0; pg < P; ++pg) {
          mma_bf16_16816(s[pg][nt], a[pg][0], a[pg][1], a[pg][2], a[pg][3], b0, b1);
          mma_bf16_16816(s[pg][nt + 1], a[pg][0], a[pg][1], a[pg][2], a[pg][3], b2, b3);
        }
      } else {
        uint32_t b0, b1;
        const int qrow = nt * 8 + (lane & 7);
        ldmatrix_x2(q_base + qrow * kRow + (2 * ks + ((lane >> 3) & 1)) * 16, b0, b1);
#pragma unroll
        for (int pg = 0; pg < P; ++pg)
          mma_bf16_16816(s[pg][nt], a[pg][0], a[pg][1], a[pg][2], a[pg][3], b0, b1);
      }
    }
  }
}

// Online-softmax update with the P tiles' log2-unit logits x (masked entries
// -inf), then O^T += V^T P^T over the P pages.  The running max starts at a
// finite kEmptyMax, so 2^(x - m) needs no guard: a masked x gives 0.
template <int D, int NT, int P, class Tile>
__device__ __forceinline__ void tile_softmax_pv(WarpState<D, NT>& st, const float (&x)[P][NT][4],
                                                const uint32_t (&v_base)[P]) {
  const int lane = threadIdx.x & 31;
  bool need = false;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float mx = fmaxf(x[0][nt][e], x[0][nt][2 + e]);
#pragma unroll
      for (int pg = 1; pg < P; ++pg) mx = fmaxf(mx, fmaxf(x[pg][nt][e], x[pg][nt][2 + e]));
      need |= mx > st.m[nt][e] + kRescaleSlack;
    }
  if (__any_sync(0xffffffffu, need)) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float mx = fmaxf(x[0][nt][e], x[0][nt][2 + e]);
#pragma unroll
        for (int pg = 1; pg < P; ++pg) mx = fmaxf(mx, fmaxf(x[pg][nt][e], x[pg][nt][2 + e]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float mnew = fmaxf(st.m[nt][e], mx);
        const float alpha = ex2(st.m[nt][e] - mnew);
        st.m[nt][e] = mnew;
        st.l[nt][e] *= alpha;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
          st.o[mt][nt][e] *= alpha;
          st.o[mt][nt][2 + e] *= alpha;
        }
      }
  }
  uint32_t pb[P][NT][2];
#pragma unroll
  for (int pg = 0; pg < P; ++pg)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float p[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) p[i] = ex2(x[pg][nt][i] - st.m[nt][i & 1]);
      st.l[nt][0] += p[0] + p[2];
      st.l[nt][1] += p[1] + p[3];
      pb[pg][nt][0] = movmatrix_trans(pack_bf16x2(p[0], p[1]));
      pb[pg][nt][1] = movmatrix_trans(pack_bf16x2(p[2], p[3]));
    }
  const int mi = lane >> 3;
  const int prow = (lane & 7) + 8 * (mi >> 1);
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) {
#pragma unroll
    for (int pg = 0; pg < P; ++pg) {
      uint32_t a0, a1, a2, a3;
      ldmatrix_x4_trans(Tile::addr(v_base[pg], prow, 2 * mt + (mi & 1)), a0, a1, a2, a3);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        mma_bf16_16816(st.o[mt][nt], a0, a1, a2, a3, pb[pg][nt][0], pb[pg][nt][1]);
    }
  }
}

// Sum each column's partial row sum over the 8 lanes sharing it.
template <int D, int NT>
__device__ __forceinline__ void reduce_row_sums(WarpState<D, NT>& st) {
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float v = st.l[nt][e];
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      st.l[nt][e] = v;
    }
}

// ---------------------------------------------------------------------------
// Combining partial softmax states (flash-decoding merge): for parts s with
// running max m_s (log2 units), sum l_s and unnormalised O_s,
//   M = max_s m_s,  f_s = 2^(m_s - M),  l = sum f_s l_s,  O = sum f_s O_s / l.
// A part with m_s = -inf has no attended position and weight 0.
// ---------------------------------------------------------------------------

// Stages one warp's O^T fragments as rows [n][D+4] (fp32) at cO + slot.
template <int D, int NT>
__device__ __forceinline__ void stage_warp_o(const WarpState<D, NT>& st, float* cO, int slot) {
  constexpr int NPAD = NT * 8;
  constexpr int OS = D + 4;
  const int lane = threadIdx.x & 31;
  const int r = lane >> 2, c = 2 * (lane & 3);
  float* ow = cO + (size_t)slot * NPAD * OS;
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int n = nt * 8 + c + (i & 1);
        const int dim = mt * 16 + r + 8 * (i >> 1);
        ow[n * OS + dim] = st.o[mt][nt][i];
      }
}

}  // namespace vegas
