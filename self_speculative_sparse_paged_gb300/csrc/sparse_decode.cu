// Sparse draft-decode attention: one draft step over the selected positions.
//
// "Vegas: Self-Speculative Decoding with Verification-Guided Sparse
// Attention", gist.science technical summary: §2 "Core mechanism" (the draft
// phase attends only to the critical KV entries selected from the previous
// verification) and §3 "Implementation" (PagedAttention with a page size of
// one token, the selected token indices passed as page indices).
//
// Here the selected positions stay logical token positions: each is mapped
// through the block table of the 16-token paged cache, so the same cache
// serves verify and draft.  One thread-block cluster of CL CTAs per
// (KV head, sequence); CTA r owns a contiguous range of the unit's list
// "T then tail".  It first resolves every entry of its range to a cache row
// (position -> page -> row) in shared memory, then each warp gathers 16-entry
// groups with one 1-D bulk copy per K row and per V row (lanes 0-15 K, 16-31
// V) into padded rows and runs the same warp core as the verify kernel with
// the G query heads of the group as the tile's columns.  The CTAs' softmax
// states meet in distributed shared memory: each CTA pushes the slices of its
// state to the CTAs that own them, then merges and writes the slice it owns,
// with no global scratch and no second pass.
#include <cooperative_groups.h>

#include "kernels.h"
#include "split_merge.cuh"

namespace cg = cooperative_groups;

namespace vegas {

template <int D, int NT>
struct SparseCfg {
  // Warps, each with two 16-row groups in flight: sixteen at head_dim 64 (a
  // group is half the bytes of a head_dim-128 one; 3% faster than eight warps
  // with four groups), twelve at head_dim 128 with one column tile (3% faster
  // than eight with three), eight with two column tiles (the shared memory
  // holds no more there).  More warps keep the same bytes in flight with more
  // groups computed at once.
  static constexpr int kWarps = D == 64 ? 16 : (NT == 1 ? 12 : kAttnWarps);
  static constexpr int kStages = 2;
  static constexpr int kRow = D * 2 + 16;           // padded row stride
  static constexpr int kTile = 16 * kRow;
  static constexpr int kStage = 2 * kTile;
  static constexpr int kMaxRows = kMaxSparseRowsPerCta;
  static constexpr size_t kStageBytes = size_t(kWarps) * kStages * kStage;
};

template <int D, int NT>
constexpr size_t sparse_smem_layout_bytes() {
  using Cfg = SparseCfg<D, NT>;
  return Cfg::kStageBytes                                          // stages
         + size_t(NT) * 8 * (2 * D + 16)                           // Q tile
         + (size_t(Cfg::kWarps) * Cfg::kStages + 1) * 8            // mbarriers (+ receive)
         + size_t(Cfg::kMaxRows) * 4                               // row table
         + size_t(NT) * 8 * (D + 2) * 4                            // CTA partial
         + (size_t(NT) * 8 * D + 4 * kMaxSparseCluster) * 4 + 16   // received output slices
         + size_t(kMaxSparseCluster) * NT * 8 * 2 * 4              // received m, l
         + 1024;
}
static_assert(sparse_smem_layout_bytes<128, 1>() <= 227 * 1024 &&
                  sparse_smem_layout_bytes<128, 2>() <= 227 * 1024 &&
                  sparse_smem_layout_bytes<64, 1>() <= 227 * 1024 &&
                  sparse_smem_layout_bytes<64, 2>() <= 227 * 1024,
              "shared memory of a draft CTA");

template <int D, int NT>
__global__ void __launch_bounds__(SparseCfg<D, NT>::kWarps * 32, 1)
    sparse_decode_kernel(const SparseParams p) {
  constexpr int W = SparseCfg<D, NT>::kWarps;
  constexpr int NTH = W * 32;
  constexpr int NPAD = NT * 8;
  constexpr int STAGES = SparseCfg<D, NT>::kStages;
  constexpr int ROW = SparseCfg<D, NT>::kRow;
  constexpr int TILE = SparseCfg<D, NT>::kTile;
  constexpr int STAGE = SparseCfg<D, NT>::kStage;
  constexpr int QROW = 2 * D + 16;
  using Tile = PaddedTile<D>;

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int CL = (int)cluster.num_blocks();

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* stage_area = smem;
  uint8_t* qs = smem + SparseCfg<D, NT>::kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(qs + NPAD * QROW);
  uint64_t* recv_bar = bars + W * STAGES;   // completes when every peer's state has landed
  int32_t* rows = reinterpret_cast<int32_t*>(recv_bar + 1);
  const int nel = p.group * D;              // output elements of the unit (G x D)
  const int per = ((nel + CL - 1) / CL + 3) & ~3;   // CTA r owns [r * per, (r + 1) * per); 4 | per
  if (threadIdx.x == 0) {
    // Every CTA sends this one its slice of the partial output and its G row
    // maxima and sums: 4 * CL * (slice + 2G) bytes, counted by st.async.
    mbar_init(smem_u32(recv_bar), 1);
    const int mine = max(0, min(per, nel - rank * per));
    mbar_arrive_expect_tx(smem_u32(recv_bar), uint32_t(4 * CL * (mine + 2 * p.group)));
    fence_mbar_init();
  }
  // First phase of the cluster barrier: this CTA has started and its receive
  // barrier is set up (its shared memory may receive other CTAs' stores once
  // every CTA has arrived).
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  griddep_begin();
  float* pM = reinterpret_cast<float*>(rows + SparseCfg<D, NT>::kMaxRows);   // [NPAD] CTA partial
  float* pL = pM + NPAD;                                                 // [NPAD]
  float* pO = pL + NPAD;                                                 // [NPAD][D]
  // [CL][per] output slices received (16-byte aligned: they arrive in 16-byte stores;
  // CL * per <= G * D + 4 * CL - 1)
  float* rO = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(pO + NPAD * D) + 15) &
                                       ~uintptr_t(15));
  float* rM = rO + NPAD * D + 4 * kMaxSparseCluster;   // [CL][NPAD] maxima received
  float* rL = rM + kMaxSparseCluster * NPAD;     // [CL][NPAD] row sums received

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.y, b = blockIdx.z;
  const int unit = b * p.hkv + g;
  const int cap = p.max_pages * 16;

  // The selected positions of this CTA's range are requested together with
  // k_b and the tail (entries past k_b are replaced below), so the index and
  // length loads take one round trip.
  constexpr int kPer = (SparseCfg<D, NT>::kMaxRows + NTH - 1) / NTH;   // entries a thread
  const int rbeg = rank * p.rows_per_split;
  int pos[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int i = tid + u * NTH, e = rbeg + i;
    pos[u] = (i < p.rows_per_split && e < p.k_max) ? __ldcg(&p.idx[size_t(unit) * p.k_max + e]) : 0;
  }
  int kb = p.k_per_seq[b];
  if (kb < 0 || kb > p.k_max) {
    if (tid == 0 && g == 0 && rank == 0) set_error(p.err, kErrDeviceFault);
    kb = max(0, min(kb, p.k_max));
  }
  const int tstart = p.tail_start[b];
  const int tlen = max(0, p.tail_len[b]);
  const int total = kb + tlen;
  const int rend = min(rbeg + p.rows_per_split, total);
  const int nrows = max(0, rend - rbeg);

  // The draft queries are requested with the indices and lengths, so their
  // load overlaps the block-table loads below (one 16-byte chunk per thread).
  constexpr int QCH = NPAD * (D / 8);
  static_assert(QCH <= NTH, "one Q chunk per thread");
  uint4 qchunk = make_uint4(0, 0, 0, 0);
  if (tid < QCH && tid / (D / 8) < p.group)
    qchunk = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p.q) +
                                            (size_t(b) * p.hq + g * p.group + tid / (D / 8)) * D)
        [tid % (D / 8)];

  if (tid == 0) {
    // one arrival per lane per stage use: each lane's cp.async copies signal it
    for (int i = 0; i < W * STAGES; ++i) mbar_init(smem_u32(&bars[i]), 32);
    fence_mbar_init();
  }
  // Entry e of the list: T[e] for e < k_b, else tail_start + (e - k_b).
  // Resolved in batches: every index of a thread (loaded above), then every
  // page load.
  {
    int phys[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int i = tid + u * NTH;
      const int e = rbeg + i;
      if (i >= nrows) pos[u] = 0;
      else if (e >= kb) pos[u] = tstart + (e - kb);
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      if (pos[u] < 0 || pos[u] >= cap) {
        set_error(p.err, kErrDeviceFault);
        pos[u] = 0;
      }
      phys[u] = tid + u * NTH < nrows ? __ldg(&p.block_table[size_t(b) * p.max_pages + (pos[u] >> 4)]) : 0;
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int i = tid + u * NTH;
      if (i < nrows) {
        if (phys[u] < 0 || phys[u] >= p.num_pages) {
          set_error(p.err, kErrDeviceFault);
          phys[u] = 0;
        }
        rows[i] = (phys[u] * p.hkv + g) * 16 + (pos[u] & 15);
      }
    }
  }
  if (tid < QCH)
    *reinterpret_cast<uint4*>(qs + (tid / (D / 8)) * QROW + (tid % (D / 8)) * 16) = qchunk;
  __syncthreads();

  const int ngroups = (nrows + 15) / 16;
  const int nmy = warp < ngroups ? (ngroups - warp + W - 1) / W : 0;
  const uint32_t stage0 = smem_u32(stage_area + warp * STAGES * STAGE);
  const uint32_t bar0 = smem_u32(&bars[warp * STAGES]);
  const __nv_bfloat16* kc = reinterpret_cast<const __nv_bfloat16*>(p.k_cache);
  const __nv_bfloat16* vc = reinterpret_cast<const __nv_bfloat16*>(p.v_cache);

  // The warp copies the group's 16 K rows and 16 V rows with 16-byte cp.async
  // (consecutive lanes cover consecutive 16-byte chunks of a row); rows past
  // the range repeat the group's first row (masked later).  Each lane then
  // arrives on the stage barrier when its own copies have landed.
  constexpr int CPR = D / 8;                       // 16-byte chunks per row
  auto issue = [&](int i) {
    const int grp = warp + i * W;
    const int s = i % STAGES;
#pragma unroll
    for (int j = 0; j < (32 * CPR) / 32; ++j) {
      const int c = lane + 32 * j;                 // chunk of the 32 rows (K rows, then V rows)
      const int r32 = c / CPR, cc = c % CPR;
      const int r = r32 & 15;
      const int li = grp * 16 + r;
      const int row = rows[li < nrows ? li : grp * 16];
      const __nv_bfloat16* src = (r32 < 16 ? kc : vc) + size_t(row) * D + cc * 8;
      cp_async16(stage0 + s * STAGE + (r32 < 16 ? 0 : TILE) + r * ROW + cc * 16, src);
    }
    cp_async_arrive_noinc(bar0 + s * 8);
  };
  for (int i = 0; i < min(STAGES, nmy); ++i) issue(i);

  uint32_t qf[D / 16][NT][2];
  load_q_frags<D, NT>(smem_u32(qs), qf);
  WarpState<D, NT> st;
  st.init();

  int done = 0;
  bool ok = true;
  for (; done < nmy; ++done) {
    const int i = done;
    const int s = i % STAGES;
    if (!mbar_wait_bounded(bar0 + s * 8, (i / STAGES) & 1)) {
      ok = false;
      break;
    }
    const int grp = warp + i * W;
    const uint32_t kb_s[1] = {stage0 + s * STAGE};
    const uint32_t vb_s[1] = {stage0 + s * STAGE + TILE};
    float sc[1][NT][4];
    tile_scores<D, NT, 1, Tile>(kb_s, qf, sc);
    float x[1][NT][4];
    const int valid = nrows - grp * 16;   // rows of this group inside the range
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int r = (lane >> 2) + 8 * (k >> 1);
        const int n = nt * 8 + 2 * (lane & 3) + (k & 1);
        x[0][nt][k] = (r < valid && n < p.group) ? sc[0][nt][k] * p.scale_log2 : -INFINITY;
      }
    tile_softmax_pv<D, NT, 1, Tile>(st, x, vb_s);
    __syncwarp();
    if (i + STAGES < nmy) {
      fence_proxy_async_smem();
      issue(i + STAGES);
    }
  }
  if (!ok) {
    if (lane == 0) set_error(p.err, kErrDeviceTimeout);
    for (int j = done; j < min(done + STAGES, nmy); ++j)
      (void)mbar_wait_bounded(bar0 + (j % STAGES) * 8, (j / STAGES) & 1);
  }
  reduce_row_sums<D, NT>(st);
  __syncthreads();
  cta_merge_to_smem<D, NT, W>(st, stage_area, SparseCfg<D, NT>::kStageBytes, p.group, pM, pL, pO);
  __syncthreads();   // the pushes below read elements other threads merged

  // Cluster merge: CTA r owns the output elements [r * per, (r + 1) * per) of
  // the G x D (per a multiple of four).  Every CTA pushes the slices of its
  // state to their owners' receive areas with asynchronous distributed-
  // shared-memory stores, 16 bytes each (four elements of one owner), and its
  // G row maxima and sums to every CTA, one (CTA, row) pair a thread; each
  // store counts against the owner's receive barrier, and an owner merges as
  // soon as that barrier has counted every byte it expects:
  // M = max_r m_r, O = sum_r 2^(m_r - M) O_r / sum_r 2^(m_r - M) l_r.
  // Spreading the pushes over the threads (rather than one thread a row
  // looping over the CTAs, four bytes a store) took the batch-1 step from
  // 5.75 to 5.3 us.  The receive areas are used by nothing else, so only the
  // barrier phase begun at entry (every CTA has started, its receive barrier
  // is ready) precedes the stores, and no cluster barrier follows them.
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  {
    const uint32_t rO_s = smem_u32(rO), rM_s = smem_u32(rM), rL_s = smem_u32(rL);
    const uint32_t rb = smem_u32(recv_bar);
    for (int e = 4 * tid; e < nel; e += 4 * NTH) {   // 4 | nel (D is 64 or 128)
      const int owner = e / per;                      // e .. e + 3 share it
      st_async_f32x4(cluster_map(rO_s + 4 * (rank * per + e - owner * per), owner), pO[e],
                     pO[e + 1], pO[e + 2], pO[e + 3], cluster_map(rb, owner));
    }
    static_assert(kMaxSparseCluster * 16 <= NTH, "one (CTA, row) pair a thread");
    const int t = NTH - 1 - tid;   // the last threads, which carry fewer elements
    if (t < CL * p.group) {        // CL * G <= 256 <= NTH
      const int r = t / p.group, n = t - r * p.group;
      st_async_f32(cluster_map(rM_s + 4 * (rank * NPAD + n), r), pM[n], cluster_map(rb, r));
      st_async_f32(cluster_map(rL_s + 4 * (rank * NPAD + n), r), pL[n], cluster_map(rb, r));
    }
  }
  if (!mbar_wait_cluster_bounded(smem_u32(recv_bar), 0)) {
    if (tid == 0) set_error(p.err, kErrDeviceTimeout);
    return;
  }
  {
    constexpr int R = kMaxSparseCluster;
    const int e0 = rank * per, e1 = min(nel, e0 + per);
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
    for (int e = e0 + tid; e < e1; e += NTH) {
      const int n = e / D;
      float mr[R], lr[R], v[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        mr[r] = -INFINITY;
        lr[r] = v[r] = 0.f;
        if (r < CL) {
          mr[r] = rM[r * NPAD + n];
          lr[r] = rL[r * NPAD + n];
          v[r] = rO[r * per + e - e0];
        }
      }
      float M = -INFINITY;
#pragma unroll
      for (int r = 0; r < R; ++r) M = fmaxf(M, mr[r]);
      float L = 0.f, a = 0.f;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float f = r < CL ? ex2(mr[r] - M) : 0.f;
        L += f * lr[r];
        a += f * v[r];
      }
      out[(size_t(b) * p.hq + g * p.group + n) * D + (e % D)] =
          __float2bfloat16_rn(L > 0.f ? a / L : 0.f);
    }
  }
}

// Launches, or with `clusters` set, reports how many clusters of p.num_splits
// CTAs can be resident at once.
template <int D, int NT>
static cudaError_t launch_sparse_one(const SparseParams& p, int batch, cudaStream_t stream,
                                     int* clusters = nullptr) {
  constexpr size_t smem = sparse_smem_layout_bytes<D, NT>();
  static std::atomic<uint32_t> configured{0};
  cudaError_t e = once_per_device(configured, [] {
    cudaError_t r = cudaFuncSetAttribute(sparse_decode_kernel<D, NT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (r != cudaSuccess) return r;
    return cudaFuncSetAttribute(sparse_decode_kernel<D, NT>,
                                cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  });
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.num_splits, p.hkv, batch);
  cfg.blockDim = dim3(SparseCfg<D, NT>::kWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.num_splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = clusters ? 1 : 2;
  if (clusters) return cudaOccupancyMaxActiveClusters(clusters, sparse_decode_kernel<D, NT>, &cfg);
  return cudaLaunchKernelEx(&cfg, sparse_decode_kernel<D, NT>, p);
}

static cudaError_t launch_sparse_any(const SparseParams& p, int head_dim, int ntiles, int batch,
                                     cudaStream_t stream, int* clusters) {
  if (p.num_splits < 1 || p.num_splits > kMaxSparseCluster) return cudaErrorInvalidValue;
  if (head_dim == 128) {
    if (ntiles == 1) return launch_sparse_one<128, 1>(p, batch, stream, clusters);
    if (ntiles == 2) return launch_sparse_one<128, 2>(p, batch, stream, clusters);
  } else if (head_dim == 64) {
    if (ntiles == 1) return launch_sparse_one<64, 1>(p, batch, stream, clusters);
    if (ntiles == 2) return launch_sparse_one<64, 2>(p, batch, stream, clusters);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_sparse(const SparseParams& p, int head_dim, int ntiles, int batch,
                          cudaStream_t stream) {
  return launch_sparse_any(p, head_dim, ntiles, batch, stream, nullptr);
}

int sparse_max_active_clusters(int head_dim, int ntiles, int cluster) {
  if (cluster < 1 || cluster > kMaxSparseCluster || ntiles < 1 || ntiles > 2) return 0;
  constexpr int kDevices = 32;
  // [device][head_dim 64/128][ntiles][cluster]: 0 unknown, -1 none, else the count
  static std::atomic<int> cache[kDevices][2][3][kMaxSparseCluster + 1];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevices) return 0;
  std::atomic<int>& slot = cache[dev][head_dim == 128 ? 1 : 0][ntiles][cluster];
  int c = slot.load(std::memory_order_acquire);
  if (c == 0) {
    SparseParams p{};
    p.hkv = 1;
    p.num_splits = cluster;
    int n = 0;
    if (launch_sparse_any(p, head_dim, ntiles, 1, 0, &n) != cudaSuccess) {
      (void)cudaGetLastError();
      n = 0;
    }
    c = n > 0 ? n : -1;
    slot.store(c, std::memory_order_release);
  }
  return c > 0 ? c : 0;
}

}  // namespace vegas
