// Host-side launch interface of the Vegas kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/vegas.h"

namespace vegas {

constexpr int kAttnWarps = 8;          // warps per attention CTA
constexpr int kMaxSplits = 128;        // split-KV partials per (sequence, KV head)
constexpr int kMaxSparseCluster = 16;  // CTAs per (sequence, KV head) in the draft kernel
constexpr int kMaxSparseRowsPerCta = 2048;

struct VerifyParams {
  const void* q;            // bf16 [B][T][Hq][D]
  void* out;                // bf16 [B][T][Hq][D]
  float* scores;            // fp32 [B][Hkv][score_stride] or null
  const int32_t* ctx_lens;  // [B]
  const int32_t* block_table;
  int score_stride;
  int num_pages;
  int max_pages;
  int hq, hkv, group, gamma, nq;
  uint32_t row_mask;        // capture rows: bit t set -> window row t is captured
  float* raw;               // raw-logit mode (no fused capture): fp32 [B][R][Hq][raw_stride], or null
  int raw_stride;
  int raw_rows;             // R = captured rows (popcount of row_mask) in raw mode
  float scale;              // softmax scale (logit units)
  float scale_log2;         // scale * log2(e)
  int pages_per_split;
  int num_splits;
  int cluster_merge;        // tcgen05 kernel: a unit's splits form clusters that merge on chip
  int cluster_size;         // CTAs per cluster (S); num_splits / S clusters per unit, merged
                            // across clusters through the workspace when more than one
  int* tickets;
  float* part_ml;
  float* part_o;
  int* err;
};

struct SparseParams {
  const void* q;            // bf16 [B][Hq][D]
  void* out;                // bf16 [B][Hq][D]
  const void* k_cache;      // bf16 [pages][Hkv][16][D]
  const void* v_cache;
  const int32_t* block_table;
  const int32_t* idx;       // [B][Hkv][k_max]
  const int32_t* k_per_seq;
  const int32_t* tail_start;
  const int32_t* tail_len;
  int k_max;
  int num_pages, max_pages;
  int hq, hkv, group;
  float scale_log2;
  int rows_per_split;       // list entries per CTA of the cluster
  int num_splits;           // CTAs per cluster (one cluster per unit)
  int* err;
};

struct SelectParams {
  const float* scores;
  const int32_t* ctx_lens;
  const int32_t* k_per_seq;
  int32_t* out_idx;
  int score_stride;
  int hkv;
  int k_max;
  int chunk;                // keys per CTA of a cluster: 1, 2, 4 or 8 x select_chunk_quantum()
  int shared;               // 1: one T per sequence from the sum over its KV heads
  int* err;
};

struct WindowParams {
  const int32_t* ctx_lens;
  int32_t* k_out;           // [B]
  int32_t* out_idx;         // [B][Hkv][k_max]
  int num_sink, window, hkv, k_max;
  int* err;
};

struct RawAggParams {
  const float* raw;         // [B][R][Hq][raw_stride]
  float* scores;            // [B][Hkv][score_stride]
  const int32_t* ctx_lens;
  int raw_stride, score_stride, rows, hq, hkv;
  int* err;
};

// Runs f() (a kernel-attribute setter, which acts on the current device) once
// per device: `done` holds one bit per device ordinal below 32.  Two threads
// racing on a device may both run f, which is harmless for attribute setters.
template <class F>
inline cudaError_t once_per_device(std::atomic<uint32_t>& done, F&& f) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint32_t bit = (dev >= 0 && dev < 32) ? (1u << dev) : 0u;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = f();
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Records `msg` as this host thread's vegas_last_error_detail(); returns status.
int record_failure(int status, const char* msg);

// Supplies a library-owned verify workspace (address and size) on the current device.
using ScratchFn = vegas_status_t (*)(void** workspace, size_t* bytes);
// vegas_verify_attn_capture; when `scratch` is given and the shape needs a
// workspace, it is asked for one only after every argument has been checked,
// and the workspace's counters are cleared on the stream before the launch.
vegas_status_t verify_two_rows(const vegas_paged_kv_t* kv, const void* q, void* out,
                               float* scores, int score_stride, const int32_t* ctx_lens,
                               int batch, int gamma, int capture_row_a, int capture_row_b,
                               float softmax_scale, void* workspace, size_t workspace_bytes,
                               void* stream, ScratchFn scratch);

// Shared-memory bytes and launch of each kernel; return cudaError_t.

// Largest 8-row query tile count per head_dim (d=128: 48 rows, d=64: 64 rows).
inline int verify_max_ntiles(int head_dim) { return head_dim == 128 ? 6 : 8; }
// tcgen05 verify kernel.  Its softmax handles the nq = (gamma+1)*G query
// columns rounded up to 8 (at most 40 at head_dim 128, 64 at head_dim 64); with
// capture, the two summed-query columns follow them in the MMA (N = 16, 32 or
// 64 columns in all).
inline int verify_tc_mma_columns(int nq, bool capture) {
  const int need = (nq + 7) / 8 * 8 + (capture ? 2 : 0);
  return need <= 16 ? 16 : need <= 32 ? 32 : need <= 64 ? 64 : 0;
}
inline bool verify_tc_supported(int head_dim, int nq, bool capture) {
  const int nqc = (nq + 7) / 8 * 8;
  return nq >= 1 && verify_tc_mma_columns(nq, capture) > 0 &&
         nqc <= (head_dim == 128 ? 40 : 64);
}
constexpr int kTcPagesPerTile = 8;
constexpr int kMaxVerifyCluster = 16;   // splits merged on chip (non-portable cluster size)
cudaError_t launch_verify_tc_d64(const CUtensorMap& kmap, const CUtensorMap& vmap,
                                 const VerifyParams& p, bool capture, int batch,
                                 cudaStream_t stream);
cudaError_t launch_verify_tc_d128(const CUtensorMap& kmap, const CUtensorMap& vmap,
                                  const VerifyParams& p, bool capture, int batch,
                                  cudaStream_t stream);
inline cudaError_t launch_verify_tc(const CUtensorMap& kmap, const CUtensorMap& vmap,
                                    const VerifyParams& p, int head_dim, bool capture, int batch,
                                    cudaStream_t stream) {
  return head_dim == 64 ? launch_verify_tc_d64(kmap, vmap, p, capture, batch, stream)
                        : launch_verify_tc_d128(kmap, vmap, p, capture, batch, stream);
}
// Clusters of `cluster` CTAs of the tcgen05 kernel resident at once (0: none / error).
int verify_tc_max_active_clusters_d64(int nq, bool capture, int cluster);
int verify_tc_max_active_clusters_d128(int nq, bool capture, int cluster);
inline int verify_tc_max_active_clusters(int head_dim, int nq, bool capture, int cluster) {
  return head_dim == 64 ? verify_tc_max_active_clusters_d64(nq, capture, cluster)
                        : verify_tc_max_active_clusters_d128(nq, capture, cluster);
}
template <int D, bool CAP>
cudaError_t launch_verify_t(const CUtensorMap& kmap, const CUtensorMap& vmap,
                            const VerifyParams& p, int ntiles, int batch, cudaStream_t stream);

size_t sparse_smem_bytes(int head_dim, int ntiles);
// Clusters of `cluster` draft-kernel CTAs resident at once (0: none / error).
int sparse_max_active_clusters(int head_dim, int ntiles, int cluster);
cudaError_t launch_sparse(const SparseParams& p, int head_dim, int ntiles, int batch,
                          cudaStream_t stream);

cudaError_t launch_select_window(const WindowParams& p, int batch, cudaStream_t stream);
cudaError_t launch_raw_aggregate(const RawAggParams& p, int batch, int max_len,
                                 cudaStream_t stream);
int select_max_chunk();
int select_chunk_quantum();   // a CTA's chunk is a multiple of this
cudaError_t launch_select(const SelectParams& p, int cluster, int batch, cudaStream_t stream);

// One CTA waits on an mbarrier nothing arrives on, bounded by limit_ns; on
// running out it records kErrDeviceTimeout in *err and writes 0 to *outcome.
cudaError_t launch_bounded_wait_check(unsigned long long limit_ns, int* err, int* outcome,
                                      cudaStream_t stream);

cudaError_t launch_synth_kv(void* cache, int which, uint64_t seed, int layer, const int32_t* owner,
                            int num_pages, int hkv, int head_dim, int max_pages,
                            const int32_t* ctx_lens, const int32_t* positions,
                            uint64_t heavy_threshold, int heavy_last, const float* unit_dir,
                            cudaStream_t stream);

}  // namespace vegas
