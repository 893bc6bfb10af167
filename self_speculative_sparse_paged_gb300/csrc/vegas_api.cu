// C ABI of the Vegas hot path: host-side validation, launch configuration,
// TMA descriptors and the device error word.  Declarations and contracts are
// in include/vegas.h and include/vegas_synth.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/vegas.h"
#include "../../include/vegas_synth.h"
#include "kernels.h"

#define VEGAS_API extern "C" __attribute__((visibility("default")))

namespace {

__device__ int g_error_word;   // one per device; kernels record the first fault here

thread_local char g_detail[512] = "";

vegas_status_t fail(vegas_status_t st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_detail, sizeof(g_detail), fmt, ap);
  va_end(ap);
  return st;
}

vegas_status_t cuda_fail(cudaError_t e, const char* where) {
  return fail(VEGAS_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;
std::mutex g_mu;   // serialises the first lookup per device only
std::atomic<int*> g_err_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};   // written before g_err_ptr[dev] is published

// Device address of the error word and SM count of the current device (looked
// up once per device; later calls take no lock).
vegas_status_t device_info(int** err, int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(VEGAS_ERR_UNSUPPORTED, "device ordinal %d", dev);
  int* ep = g_err_ptr[dev].load(std::memory_order_acquire);
  if (!ep) {
    std::lock_guard<std::mutex> lock(g_mu);
    ep = g_err_ptr[dev].load(std::memory_order_relaxed);
    if (!ep) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_error_word);
      if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
      int n = 0;
      e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
      g_sms[dev] = n;
      ep = static_cast<int*>(p);
      g_err_ptr[dev].store(ep, std::memory_order_release);
    }
  }
  if (err) *err = ep;
  if (sms) *sms = g_sms[dev];
  return VEGAS_OK;
}


// ----------------------------------------------------------------- TMA maps
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

vegas_status_t get_encoder(EncodeTiledFn* fn) {
  static EncodeTiledFn cached = nullptr;
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                           &q);
    if (err == cudaSuccess && q == cudaDriverEntryPointSuccess) cached = (EncodeTiledFn)p;
  });
  if (!cached) return fail(VEGAS_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (%s)",
                           cudaGetErrorString(err));
  *fn = cached;
  return VEGAS_OK;
}

// 2-D view of a paged cache: rows = num_pages * Hkv * 16, head_dim bf16 each;
// box 16 rows x 64 elements (128 bytes), 128-byte swizzle.
vegas_status_t make_cache_map(CUtensorMap* map, const void* base, const vegas_paged_kv_t* kv) {
  EncodeTiledFn enc;
  vegas_status_t st = get_encoder(&enc);
  if (st != VEGAS_OK) return st;
  cuuint64_t dims[2] = {(cuuint64_t)kv->head_dim,
                        (cuuint64_t)kv->num_pages * kv->num_kv_heads * VEGAS_PAGE_SIZE};
  cuuint64_t strides[1] = {(cuuint64_t)kv->head_dim * 2};
  cuuint32_t box[2] = {64, 16};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(VEGAS_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return VEGAS_OK;
}

// ----------------------------------------------------------------- checks
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

vegas_status_t check_kv(const vegas_paged_kv_t* kv) {
  if (!kv) return fail(VEGAS_ERR_INVALID_ARG, "kv is NULL");
  if (!kv->k_cache || !kv->v_cache || !kv->block_table)
    return fail(VEGAS_ERR_INVALID_ARG, "kv: NULL cache or block table");
  if (!aligned16(kv->k_cache) || !aligned16(kv->v_cache))
    return fail(VEGAS_ERR_INVALID_ARG, "kv: caches must be 16-byte aligned");
  if (kv->page_size != VEGAS_PAGE_SIZE)
    return fail(VEGAS_ERR_UNSUPPORTED, "page_size %d (only 16)", kv->page_size);
  if (kv->head_dim != 64 && kv->head_dim != 128)
    return fail(VEGAS_ERR_UNSUPPORTED, "head_dim %d (64 or 128)", kv->head_dim);
  if (kv->num_kv_heads < 1 || kv->num_q_heads < 1 || kv->num_q_heads % kv->num_kv_heads)
    return fail(VEGAS_ERR_INVALID_ARG, "heads: Hq %d must be a positive multiple of Hkv %d",
                kv->num_q_heads, kv->num_kv_heads);
  if (kv->num_pages < 1 || kv->max_pages_per_seq < 1)
    return fail(VEGAS_ERR_INVALID_ARG, "num_pages %d / max_pages_per_seq %d", kv->num_pages,
                kv->max_pages_per_seq);
  if ((long long)kv->num_pages * kv->num_kv_heads * VEGAS_PAGE_SIZE >= (1ll << 31))
    return fail(VEGAS_ERR_UNSUPPORTED, "cache rows (num_pages * Hkv * 16) must be < 2^31");
  if ((long long)kv->max_pages_per_seq * VEGAS_PAGE_SIZE >= (1ll << 24))
    return fail(VEGAS_ERR_UNSUPPORTED, "sequence capacity must be < 2^24 positions");
  return VEGAS_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Splits per (sequence, KV head): fill whole waves of one CTA per SM.
int verify_splits(int units, int max_pages, int sms) {
  const int s0 = (sms + units - 1) / units;
  int best = 1;
  double best_eff = -1.0;
  const int hi = std::min(std::min(4 * s0, vegas::kMaxSplits), std::max(1, max_pages / 8));
  for (int s = std::max(1, std::min(s0, hi)); s <= hi; ++s) {
    const long long ctas = (long long)units * s;
    const long long waves = (ctas + sms - 1) / sms;
    const double eff = double(ctas) / double(waves * sms);
    if (eff > best_eff + 1e-9) {
      best = s;
      best_eff = eff;
    }
    if (eff >= 0.999) break;
  }
  return best;
}

struct VerifyPlan {
  int nq, ncols, ntiles, splits, pages_per_split;
  bool tc;        // tcgen05 kernel instead of the mma.sync one (verify_tc_supported)
  bool cluster;   // tcgen05 kernel with a unit's splits in clusters merging on chip
  int cluster_size;   // CTAs per cluster; splits / cluster_size clusters per unit
  bool needs_ws;      // partials or tickets go through the workspace
  size_t tickets_off, ml_off, o_off, bytes;
};

// Query columns of the verify tile: the (gamma+1)*G rows, plus with capture
// two columns holding the summed captured query (at the next even index).
int verify_columns(int nq, bool capture) { return capture ? ((nq + 1) & ~1) + 2 : nq; }

VerifyPlan plan_verify(const vegas_paged_kv_t* kv, int batch, int gamma, int sms, bool capture,
                       bool with_device) {
  VerifyPlan pl{};
  const int G = kv->num_q_heads / kv->num_kv_heads;
  pl.nq = (gamma + 1) * G;
  pl.ncols = verify_columns(pl.nq, capture);
  pl.ntiles = (pl.ncols + 7) / 8;
  pl.tc = vegas::verify_tc_supported(kv->head_dim, pl.nq, capture);
  const int units = std::max(1, batch * kv->num_kv_heads);
  if (pl.tc && units < sms && with_device) {
    // C clusters of S CTAs per unit, every CTA resident (one wave), >= one tile
    // per split, as many CTAs as fit (larger clusters first on ties): a
    // cluster's splits merge through distributed shared memory, the clusters of
    // a unit through a few rows of the workspace.
    const int max_splits = std::max(1, kv->max_pages_per_seq / vegas::kTcPagesPerTile);
    int bestS = 0, bestC = 0, oneS = 0;
    for (int S = std::min(vegas::kMaxVerifyCluster, sms / units); S >= 2; --S) {
      const int resident =
          vegas::verify_tc_max_active_clusters(kv->head_dim, pl.nq, capture, S);
      if (!oneS && S <= max_splits && resident >= units) oneS = S;
      // (the cross-cluster merge takes one lane per cluster: C <= 32)
      int C = std::min(std::min(sms / (units * S), max_splits / S), 32);
      while (C > 0 && resident < units * C) --C;
      if (C > 0 && S * C > bestS * bestC) {
        bestS = S;
        bestC = C;
      }
    }
    // One cluster per unit when it already covers 60% of the SMs: more CTAs
    // measured no faster there (the stream is not what limits a launch), and
    // it needs no workspace.
    if (oneS > 1 && 10 * oneS * units >= 6 * sms) {
      bestS = oneS;
      bestC = 1;
    }
    if (bestS > 1) {
      // split s takes pages [s * max_pages / n, (s + 1) * max_pages / n): >= 8 each
      const int n = bestS * bestC;
      pl.splits = n;
      pl.pages_per_split = (kv->max_pages_per_seq + n - 1) / n;
      pl.cluster = true;
      pl.cluster_size = bestS;
      const int C = bestC;
      if (C > 1) {
        pl.needs_ws = true;
        pl.tickets_off = 0;
        pl.ml_off = align256(size_t(units) * bestS * 4);
        pl.o_off = pl.ml_off + align256(size_t(units) * C * pl.nq * 2 * 4);
        pl.bytes = pl.o_off + size_t(units) * C * pl.nq * kv->head_dim * 4;
      }
      return pl;   // bytes = 0 with one cluster per unit
    }
  }
  pl.cluster_size = 1;
  pl.splits = verify_splits(units, kv->max_pages_per_seq, sms);
  // the last-arriving tcgen05 CTA stages 3 floats per (partial, row) of its
  // unit in the freed K/V rings: at most 2 * splits * nq * 12 bytes <= 96 KB
  if (pl.tc) pl.splits = std::max(1, std::min(pl.splits, 96 * 1024 / (24 * pl.nq)));
  pl.pages_per_split = (kv->max_pages_per_seq + pl.splits - 1) / pl.splits;
  // splits cover whole tiles: 8 pages (tcgen05 kernel) or page pairs
  const int quantum = pl.tc ? vegas::kTcPagesPerTile : 2;
  pl.pages_per_split = (pl.pages_per_split + quantum - 1) / quantum * quantum;
  pl.splits = (kv->max_pages_per_seq + pl.pages_per_split - 1) / pl.pages_per_split;
  // the tcgen05 kernel leaves one partial per softmax group (two per split)
  const size_t parts = size_t(pl.splits) * (pl.tc ? 2 : 1);
  pl.tickets_off = 0;
  pl.ml_off = align256(size_t(units) * 4);
  pl.o_off = pl.ml_off + align256(size_t(units) * parts * pl.nq * 2 * 4);
  pl.bytes = pl.o_off + size_t(units) * parts * pl.nq * kv->head_dim * 4;
  pl.needs_ws = pl.splits > 1;
  return pl;
}

struct SparsePlan {
  int ntiles, cluster, rows_per_cta;
};

// One cluster per (sequence, KV head).  Few units (fewer than half the SMs):
// the largest cluster (up to 16 CTAs, each at least 64 entries of the list)
// whose clusters are all resident at once, so every SM gathers.  Many units:
// one wave of units x cluster <= SMs when every CTA's share fits its row
// table, else the fewest CTAs that fit it.
SparsePlan plan_sparse(const vegas_paged_kv_t* kv, int batch, int k_max, int max_tail, int sms) {
  SparsePlan pl{};
  const int G = kv->num_q_heads / kv->num_kv_heads;
  pl.ntiles = (G + 7) / 8;
  const int units = std::max(1, batch * kv->num_kv_heads);
  const int rows_max = std::max(1, k_max + max_tail);
  const int fit = (rows_max + vegas::kMaxSparseRowsPerCta - 1) / vegas::kMaxSparseRowsPerCta;
  int cl;
  if (2 * units < sms) {
    cl = std::min(vegas::kMaxSparseCluster, std::max(fit, std::min(sms / units,
                                                                   (rows_max + 63) / 64)));
    while (cl > std::max(fit, 1) &&
           vegas::sparse_max_active_clusters(kv->head_dim, pl.ntiles, cl) < units)
      --cl;
  } else {
    cl = std::max(fit, std::min(vegas::kMaxSparseCluster, std::max(1, sms / units)));
  }
  const int rpc = (rows_max + cl - 1) / cl;
  pl.rows_per_cta = (rpc + 15) / 16 * 16;
  pl.cluster = cl;
  return pl;
}

cudaError_t launch_verify_any(const CUtensorMap& km, const CUtensorMap& vm,
                              const vegas::VerifyParams& p, int d, int nt, bool cap, int batch,
                              cudaStream_t s) {
  if (d == 128)
    return cap ? vegas::launch_verify_t<128, true>(km, vm, p, nt, batch, s)
               : vegas::launch_verify_t<128, false>(km, vm, p, nt, batch, s);
  return cap ? vegas::launch_verify_t<64, true>(km, vm, p, nt, batch, s)
             : vegas::launch_verify_t<64, false>(km, vm, p, nt, batch, s);
}

}  // namespace

namespace vegas {
int record_failure(int status, const char* msg) {
  return (int)fail(static_cast<vegas_status_t>(status), "%s", msg);
}
}  // namespace vegas

// =========================================================================
// Verify attention with Collect-2-Query capture
// =========================================================================
VEGAS_API size_t vegas_verify_workspace_size(const vegas_paged_kv_t* kv, int batch, int gamma) {
  if (check_kv(kv) != VEGAS_OK || batch < 0 || gamma < 0) return 0;
  int sms = 0;
  const bool dev = device_info(nullptr, &sms) == VEGAS_OK && sms > 0;
  if (!dev) sms = 148;
  return std::max(plan_verify(kv, batch, gamma, sms, true, dev).bytes,
                  plan_verify(kv, batch, gamma, sms, false, dev).bytes);
}

namespace {
vegas_status_t verify_impl(const vegas_paged_kv_t* kv, const void* q, void* out, float* scores,
                           int score_stride, const int32_t* ctx_lens, int batch, int gamma,
                           uint32_t row_mask, float softmax_scale, void* workspace,
                           size_t workspace_bytes, void* stream, float* raw = nullptr,
                           int raw_stride = 0, vegas::ScratchFn scratch = nullptr);
}  // namespace

namespace vegas {
// vegas_verify_attn_capture; with `scratch`, the workspace comes from it once
// every argument has been checked, and its counters are cleared on the stream
// just before the launch.
vegas_status_t verify_two_rows(const vegas_paged_kv_t* kv, const void* q, void* out,
                               float* scores, int score_stride, const int32_t* ctx_lens,
                               int batch, int gamma, int capture_row_a, int capture_row_b,
                               float softmax_scale, void* workspace, size_t workspace_bytes,
                               void* stream, ScratchFn scratch) {
  uint32_t mask = 0;
  if (scores) {
    if (gamma < 0 || gamma > 15) return fail(VEGAS_ERR_UNSUPPORTED, "gamma %d (0..15)", gamma);
    if (capture_row_a < 0 || capture_row_a > gamma || capture_row_b < 0 || capture_row_b > gamma)
      return fail(VEGAS_ERR_INVALID_ARG, "capture rows (%d, %d) outside [0, %d]", capture_row_a,
                  capture_row_b, gamma);
    mask = (1u << capture_row_a) | (1u << capture_row_b);
  }
  return verify_impl(kv, q, out, scores, score_stride, ctx_lens, batch, gamma, mask,
                     softmax_scale, workspace, workspace_bytes, stream, nullptr, 0, scratch);
}
}  // namespace vegas

VEGAS_API vegas_status_t vegas_verify_attn_capture(
    const vegas_paged_kv_t* kv, const void* q, void* out, float* scores, int score_stride,
    const int32_t* ctx_lens, int batch, int gamma, int capture_row_a, int capture_row_b,
    float softmax_scale, void* workspace, size_t workspace_bytes, void* stream) {
  return vegas::verify_two_rows(kv, q, out, scores, score_stride, ctx_lens, batch, gamma,
                                capture_row_a, capture_row_b, softmax_scale, workspace,
                                workspace_bytes, stream, nullptr);
}

VEGAS_API vegas_status_t vegas_verify_attn_raw_logits(
    const vegas_paged_kv_t* kv, const void* q, void* out, float* raw, int raw_stride,
    const int32_t* ctx_lens, int batch, int gamma, uint32_t capture_row_mask,
    float softmax_scale, void* workspace, size_t workspace_bytes, void* stream) {
  if (!raw) return fail(VEGAS_ERR_INVALID_ARG, "NULL raw");
  if (raw_stride < 1) return fail(VEGAS_ERR_INVALID_ARG, "raw_stride %d", raw_stride);
  if (gamma < 0 || gamma > 15) return fail(VEGAS_ERR_UNSUPPORTED, "gamma %d (0..15)", gamma);
  if (capture_row_mask == 0 || (capture_row_mask >> (gamma + 1)) != 0)
    return fail(VEGAS_ERR_INVALID_ARG, "capture row mask 0x%x: needs rows in [0, %d]",
                capture_row_mask, gamma);
  return verify_impl(kv, q, out, nullptr, 0, ctx_lens, batch, gamma, capture_row_mask,
                     softmax_scale, workspace, workspace_bytes, stream, raw, raw_stride);
}

VEGAS_API vegas_status_t vegas_aggregate_raw_logits(const float* raw, int raw_stride,
                                                    const int32_t* ctx_lens, int batch,
                                                    int num_rows, int num_q_heads,
                                                    int num_kv_heads, int max_len,
                                                    float* scores, int score_stride,
                                                    void* stream) {
  if (!raw || !ctx_lens || !scores) return fail(VEGAS_ERR_INVALID_ARG, "NULL pointer argument");
  if (batch < 0 || num_rows < 1 || num_kv_heads < 1 || num_q_heads < num_kv_heads ||
      num_q_heads % num_kv_heads != 0 || raw_stride < 1 || score_stride < 1 || max_len < 0)
    return fail(VEGAS_ERR_INVALID_ARG,
                "batch %d, rows %d, heads %d/%d, strides %d/%d, max_len %d", batch, num_rows,
                num_q_heads, num_kv_heads, raw_stride, score_stride, max_len);
  if (batch == 0) return VEGAS_OK;
  int* err = nullptr;
  vegas_status_t st = device_info(&err, nullptr);
  if (st != VEGAS_OK) return st;
  vegas::RawAggParams p{};
  p.raw = raw;
  p.scores = scores;
  p.ctx_lens = ctx_lens;
  p.raw_stride = raw_stride;
  p.score_stride = score_stride;
  p.rows = num_rows;
  p.hq = num_q_heads;
  p.hkv = num_kv_heads;
  p.err = err;
  cudaError_t e = vegas::launch_raw_aggregate(p, batch, max_len, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "raw aggregate launch");
  return VEGAS_OK;
}

VEGAS_API vegas_status_t vegas_verify_attn_capture_rows(
    const vegas_paged_kv_t* kv, const void* q, void* out, float* scores, int score_stride,
    const int32_t* ctx_lens, int batch, int gamma, uint32_t capture_row_mask,
    float softmax_scale, void* workspace, size_t workspace_bytes, void* stream) {
  if (scores) {
    if (gamma < 0 || gamma > 15) return fail(VEGAS_ERR_UNSUPPORTED, "gamma %d (0..15)", gamma);
    if (capture_row_mask == 0 || (capture_row_mask >> (gamma + 1)) != 0)
      return fail(VEGAS_ERR_INVALID_ARG, "capture row mask 0x%x: needs rows in [0, %d]",
                  capture_row_mask, gamma);
  }
  return verify_impl(kv, q, out, scores, score_stride, ctx_lens, batch, gamma, capture_row_mask,
                     softmax_scale, workspace, workspace_bytes, stream);
}

namespace {
vegas_status_t verify_impl(const vegas_paged_kv_t* kv, const void* q, void* out, float* scores,
                           int score_stride, const int32_t* ctx_lens, int batch, int gamma,
                           uint32_t row_mask, float softmax_scale, void* workspace,
                           size_t workspace_bytes, void* stream, float* raw, int raw_stride,
                           vegas::ScratchFn scratch) {
  vegas_status_t st = check_kv(kv);
  if (st != VEGAS_OK) return st;
  if (batch < 0) return fail(VEGAS_ERR_INVALID_ARG, "batch %d", batch);
  if (gamma < 0 || gamma > 15) return fail(VEGAS_ERR_UNSUPPORTED, "gamma %d (0..15)", gamma);
  if (!q || !out || !ctx_lens) return fail(VEGAS_ERR_INVALID_ARG, "NULL q, out or ctx_lens");
  if (!aligned16(q) || !aligned16(out))
    return fail(VEGAS_ERR_INVALID_ARG, "q and out must be 16-byte aligned");
  if (!std::isfinite(softmax_scale)) return fail(VEGAS_ERR_INVALID_ARG, "softmax_scale not finite");
  const int G = kv->num_q_heads / kv->num_kv_heads;
  const int nq = (gamma + 1) * G;
  const int ncols = verify_columns(nq, scores != nullptr);
  if ((ncols + 7) / 8 > vegas::verify_max_ntiles(kv->head_dim))
    return fail(VEGAS_ERR_UNSUPPORTED,
                "(gamma+1)*G = %d query rows (+2 capture columns) exceeds %d for head_dim %d", nq,
                8 * vegas::verify_max_ntiles(kv->head_dim), kv->head_dim);
  if (scores && score_stride < 1)
    return fail(VEGAS_ERR_INVALID_ARG, "score_stride %d", score_stride);
  if (batch == 0) return VEGAS_OK;
  int* err = nullptr;
  int sms = 0;
  if ((st = device_info(&err, &sms)) != VEGAS_OK) return st;
  const VerifyPlan pl = plan_verify(kv, batch, gamma, sms, scores != nullptr, true);
  const bool needs_ws = pl.needs_ws;
  if (scratch) {
    // A library-owned scratch serves exactly the shapes whose reported
    // workspace size fits it, whether or not this launch would use it.
    if ((st = scratch(&workspace, &workspace_bytes)) != VEGAS_OK) return st;
    const size_t reported = std::max(plan_verify(kv, batch, gamma, sms, true, true).bytes,
                                      plan_verify(kv, batch, gamma, sms, false, true).bytes);
    if (reported > workspace_bytes)
      return fail(VEGAS_ERR_WORKSPACE_TOO_SMALL, "verify workspace %zu < %zu bytes",
                  workspace_bytes, reported);
  }
  if (needs_ws) {
    if (!workspace || workspace_bytes < pl.bytes)
      return fail(VEGAS_ERR_WORKSPACE_TOO_SMALL, "verify workspace %zu < %zu bytes",
                  workspace_bytes, pl.bytes);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
      return fail(VEGAS_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  }
  CUtensorMap km, vm;
  if ((st = make_cache_map(&km, kv->k_cache, kv)) != VEGAS_OK) return st;
  if ((st = make_cache_map(&vm, kv->v_cache, kv)) != VEGAS_OK) return st;
  vegas::VerifyParams p{};
  p.q = q;
  p.out = out;
  p.scores = scores;
  p.ctx_lens = ctx_lens;
  p.block_table = kv->block_table;
  p.score_stride = score_stride;
  p.num_pages = kv->num_pages;
  p.max_pages = kv->max_pages_per_seq;
  p.hq = kv->num_q_heads;
  p.hkv = kv->num_kv_heads;
  p.group = G;
  p.gamma = gamma;
  p.nq = nq;
  p.row_mask = row_mask;
  p.raw = raw;
  p.raw_stride = raw_stride;
  p.raw_rows = __builtin_popcount(row_mask);
  p.scale = softmax_scale;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.pages_per_split = pl.pages_per_split;
  p.num_splits = pl.splits;
  p.cluster_merge = pl.cluster ? 1 : 0;
  p.cluster_size = pl.cluster ? pl.cluster_size : 1;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.tickets = ws ? reinterpret_cast<int*>(ws + pl.tickets_off) : nullptr;
  p.part_ml = ws ? reinterpret_cast<float*>(ws + pl.ml_off) : nullptr;
  p.part_o = ws ? reinterpret_cast<float*>(ws + pl.o_off) : nullptr;
  p.err = err;
  if (needs_ws && scratch) {
    // shared scratch: its per-unit counters may hold anything from an earlier call
    const size_t tickets = size_t(batch) * kv->num_kv_heads * (pl.cluster ? pl.cluster_size : 1);
    cudaError_t e = cudaMemsetAsync(p.tickets, 0, tickets * sizeof(int),
                                    static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "clear scratch counters");
  }
  cudaError_t e =
      pl.tc ? vegas::launch_verify_tc(km, vm, p, kv->head_dim, scores != nullptr, batch,
                                      static_cast<cudaStream_t>(stream))
            : launch_verify_any(km, vm, p, kv->head_dim, pl.ntiles, scores != nullptr, batch,
                                static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "verify launch");
  return VEGAS_OK;
}
}  // namespace

// =========================================================================
// Top-k select
// =========================================================================
namespace {
vegas_status_t select_impl(const float* scores, int score_stride, const int32_t* ctx_lens,
                           const int32_t* k_per_seq, int32_t* out_idx, int batch,
                           int num_kv_heads, int k_max, bool shared, void* stream) {
  if (!scores || !ctx_lens || !k_per_seq || !out_idx)
    return fail(VEGAS_ERR_INVALID_ARG, "NULL pointer argument");
  if (batch < 0 || num_kv_heads < 1 || k_max < 0 || score_stride < 1)
    return fail(VEGAS_ERR_INVALID_ARG, "batch %d, num_kv_heads %d, k_max %d, score_stride %d",
                batch, num_kv_heads, k_max, score_stride);
  const int max_chunk = vegas::select_max_chunk();
  if ((long long)score_stride > 8ll * max_chunk)
    return fail(VEGAS_ERR_UNSUPPORTED, "score_stride %d exceeds %d", score_stride, 8 * max_chunk);
  if (batch == 0 || k_max == 0) return VEGAS_OK;
  int* err = nullptr;
  int sms = 0;
  vegas_status_t st = device_info(&err, &sms);
  if (st != VEGAS_OK) return st;
  const int units = batch * (shared ? 1 : num_kv_heads);
  const int quantum = vegas::select_chunk_quantum();
  auto chunk_for = [&](int c) {   // a power-of-two number of quanta
    const int ch = (score_stride + c - 1) / c;
    int q = quantum;
    while (q < ch) q *= 2;
    return q;
  };
  int cl = 1;
  while (chunk_for(cl) > max_chunk) cl *= 2;
  // spread small batches over more CTAs while each keeps a full quantum of keys
  while (cl < 8 && units * cl * 2 <= sms && score_stride / (2 * cl) >= quantum) cl *= 2;
  vegas::SelectParams p{};
  p.scores = scores;
  p.ctx_lens = ctx_lens;
  p.k_per_seq = k_per_seq;
  p.out_idx = out_idx;
  p.score_stride = score_stride;
  p.hkv = num_kv_heads;
  p.k_max = k_max;
  p.chunk = chunk_for(cl);
  p.shared = shared ? 1 : 0;
  p.err = err;
  cudaError_t e = vegas::launch_select(p, cl, batch, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "select launch");
  return VEGAS_OK;
}
}  // namespace

VEGAS_API vegas_status_t vegas_select_topk(const float* scores, int score_stride,
                                           const int32_t* ctx_lens, const int32_t* k_per_seq,
                                           int32_t* out_idx, int batch, int num_kv_heads,
                                           int k_max, void* stream) {
  return select_impl(scores, score_stride, ctx_lens, k_per_seq, out_idx, batch, num_kv_heads,
                     k_max, false, stream);
}

VEGAS_API vegas_status_t vegas_select_topk_shared(const float* scores, int score_stride,
                                                  const int32_t* ctx_lens,
                                                  const int32_t* k_per_seq, int32_t* out_idx,
                                                  int batch, int num_kv_heads, int k_max,
                                                  void* stream) {
  return select_impl(scores, score_stride, ctx_lens, k_per_seq, out_idx, batch, num_kv_heads,
                     k_max, true, stream);
}

VEGAS_API vegas_status_t vegas_select_window(const int32_t* ctx_lens, int num_sink, int window,
                                             int32_t* k_out, int32_t* out_idx, int batch,
                                             int num_kv_heads, int k_max, void* stream) {
  if (!ctx_lens || !k_out || !out_idx) return fail(VEGAS_ERR_INVALID_ARG, "NULL pointer argument");
  if (batch < 0 || num_kv_heads < 1 || num_sink < 0 || window < 0 ||
      (long long)num_sink + window > (1 << 30))
    return fail(VEGAS_ERR_INVALID_ARG, "batch %d, num_kv_heads %d, num_sink %d, window %d", batch,
                num_kv_heads, num_sink, window);
  if ((long long)k_max < (long long)num_sink + window)
    return fail(VEGAS_ERR_INVALID_ARG, "k_max %d < num_sink + window = %d", k_max,
                num_sink + window);
  if (batch == 0) return VEGAS_OK;
  int* err = nullptr;
  vegas_status_t st = device_info(&err, nullptr);
  if (st != VEGAS_OK) return st;
  vegas::WindowParams p{};
  p.ctx_lens = ctx_lens;
  p.k_out = k_out;
  p.out_idx = out_idx;
  p.num_sink = num_sink;
  p.window = window;
  p.hkv = num_kv_heads;
  p.k_max = k_max;
  p.err = err;
  cudaError_t e = vegas::launch_select_window(p, batch, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "window select launch");
  return VEGAS_OK;
}

// =========================================================================
// Sparse draft-decode attention
// =========================================================================
VEGAS_API vegas_status_t vegas_sparse_decode_attn(
    const vegas_paged_kv_t* kv, const void* q, void* out, const int32_t* idx, int k_max,
    const int32_t* k_per_seq, const int32_t* tail_start, const int32_t* tail_len, int max_tail,
    int batch, float softmax_scale, void* stream) {
  vegas_status_t st = check_kv(kv);
  if (st != VEGAS_OK) return st;
  if (batch < 0 || k_max < 0 || max_tail < 0)
    return fail(VEGAS_ERR_INVALID_ARG, "batch %d, k_max %d, max_tail %d", batch, k_max, max_tail);
  if (k_max + max_tail < 1) return fail(VEGAS_ERR_INVALID_ARG, "empty attention set");
  if (!q || !out || !k_per_seq || !tail_start || !tail_len || (k_max > 0 && !idx))
    return fail(VEGAS_ERR_INVALID_ARG, "NULL pointer argument");
  if (!aligned16(q)) return fail(VEGAS_ERR_INVALID_ARG, "q must be 16-byte aligned");
  if (!std::isfinite(softmax_scale)) return fail(VEGAS_ERR_INVALID_ARG, "softmax_scale not finite");
  const int G = kv->num_q_heads / kv->num_kv_heads;
  if (G > 16) return fail(VEGAS_ERR_UNSUPPORTED, "group size %d (at most 16)", G);
  if ((long long)k_max + max_tail > vegas::kMaxSparseCluster * vegas::kMaxSparseRowsPerCta)
    return fail(VEGAS_ERR_UNSUPPORTED, "k_max + max_tail = %lld exceeds %d",
                (long long)k_max + max_tail, vegas::kMaxSparseCluster * vegas::kMaxSparseRowsPerCta);
  if (batch == 0) return VEGAS_OK;
  int* err = nullptr;
  int sms = 0;
  if ((st = device_info(&err, &sms)) != VEGAS_OK) return st;
  const SparsePlan pl = plan_sparse(kv, batch, k_max, max_tail, sms);
  vegas::SparseParams p{};
  p.q = q;
  p.out = out;
  p.k_cache = kv->k_cache;
  p.v_cache = kv->v_cache;
  p.block_table = kv->block_table;
  p.idx = idx;
  p.k_per_seq = k_per_seq;
  p.tail_start = tail_start;
  p.tail_len = tail_len;
  p.k_max = k_max;
  p.num_pages = kv->num_pages;
  p.max_pages = kv->max_pages_per_seq;
  p.hq = kv->num_q_heads;
  p.hkv = kv->num_kv_heads;
  p.group = G;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.rows_per_split = pl.rows_per_cta;
  p.num_splits = pl.cluster;
  p.err = err;
  cudaError_t e = vegas::launch_sparse(p, kv->head_dim, pl.ntiles, batch,
                                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "sparse launch");
  return VEGAS_OK;
}

// =========================================================================
// Synthetic input generator
// =========================================================================
VEGAS_API vegas_status_t vegas_synth_paged_kv(void* cache, int which, uint64_t seed, int layer,
                                              const int32_t* owner, int num_pages,
                                              int num_kv_heads, int head_dim,
                                              int max_pages_per_seq, const int32_t* ctx_lens,
                                              const int32_t* positions, uint64_t heavy_threshold,
                                              int heavy_last, const float* unit_dir,
                                              void* stream) {
  if (!cache || !owner || !ctx_lens || !positions || !unit_dir)
    return fail(VEGAS_ERR_INVALID_ARG, "NULL pointer argument");
  if ((which != 0 && which != 1) || layer < 0 || num_pages < 1 || num_kv_heads < 1 ||
      (head_dim != 64 && head_dim != 128) || max_pages_per_seq < 1 || heavy_last < 0)
    return fail(VEGAS_ERR_INVALID_ARG, "bad generator shape");
  if (!aligned16(cache)) return fail(VEGAS_ERR_INVALID_ARG, "cache must be 16-byte aligned");
  cudaError_t e = vegas::launch_synth_kv(cache, which, seed, layer, owner, num_pages, num_kv_heads,
                                         head_dim, max_pages_per_seq, ctx_lens, positions,
                                         heavy_threshold, heavy_last, unit_dir,
                                         static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "synth launch");
  return VEGAS_OK;
}

// =========================================================================
// One decode iteration over a stack of layers (layer-pipelined select)
// =========================================================================
namespace {

// Events ordering select(l) between the two streams: 2 per layer, created once
// per device and reused; a device's calls enqueue one at a time.
struct EventPool {
  std::mutex mu;
  std::vector<cudaEvent_t> ev;
};
EventPool g_event_pool[kMaxDevices];

vegas_status_t check_layer(const vegas_layer_t& L, const vegas_layer_t& L0, int i) {
  vegas_status_t st = check_kv(&L.kv);
  if (st != VEGAS_OK) {
    char why[sizeof(g_detail)];
    std::snprintf(why, sizeof(why), "%s", g_detail);
    return fail(st, "layer %d: %s", i, why);
  }
  if (L.kv.num_q_heads != L0.kv.num_q_heads || L.kv.num_kv_heads != L0.kv.num_kv_heads ||
      L.kv.head_dim != L0.kv.head_dim || L.kv.max_pages_per_seq != L0.kv.max_pages_per_seq)
    return fail(VEGAS_ERR_INVALID_ARG, "layer %d: heads, head_dim or max_pages differ from layer 0",
                i);
  if (!L.q_verify || !L.out_verify || !L.q_draft || !L.out_draft || !L.scores || !L.idx)
    return fail(VEGAS_ERR_INVALID_ARG, "layer %d: NULL pointer", i);
  if (!aligned16(L.q_verify) || !aligned16(L.out_verify) || !aligned16(L.q_draft) ||
      !aligned16(L.out_draft))
    return fail(VEGAS_ERR_INVALID_ARG, "layer %d: queries and outputs must be 16-byte aligned", i);
  return VEGAS_OK;
}

}  // namespace

VEGAS_API vegas_status_t vegas_decode_iteration(
    const vegas_layer_t* layers, int num_layers, const int32_t* ctx_lens,
    const int32_t* k_per_seq, const int32_t* tail_lens, int max_tail, int batch, int gamma,
    int score_stride, int k_max, float softmax_scale, void* workspace, size_t workspace_bytes,
    void* stream, void* select_stream) {
  // ---- every check before the first launch
  if (!layers || num_layers < 1) return fail(VEGAS_ERR_INVALID_ARG, "no layers");
  if (!ctx_lens || !k_per_seq || (gamma > 0 && !tail_lens))
    return fail(VEGAS_ERR_INVALID_ARG, "NULL ctx_lens, k_per_seq or tail_lens");
  if (batch < 0 || gamma < 0 || max_tail < 0 || k_max < 1 || score_stride < 1)
    return fail(VEGAS_ERR_INVALID_ARG, "batch %d, gamma %d, max_tail %d, k_max %d, stride %d",
                batch, gamma, max_tail, k_max, score_stride);
  if (gamma > 15) return fail(VEGAS_ERR_UNSUPPORTED, "gamma %d (0..15)", gamma);
  if (!std::isfinite(softmax_scale)) return fail(VEGAS_ERR_INVALID_ARG, "softmax_scale not finite");
  if (select_stream && select_stream == stream)
    return fail(VEGAS_ERR_INVALID_ARG, "select_stream must differ from stream (or be NULL)");
  for (int i = 0; i < num_layers; ++i) {
    vegas_status_t st = check_layer(layers[i], layers[0], i);
    if (st != VEGAS_OK) return st;
  }
  const vegas_paged_kv_t& kv0 = layers[0].kv;
  const int G = kv0.num_q_heads / kv0.num_kv_heads;
  if ((verify_columns((gamma + 1) * G, true) + 7) / 8 > vegas::verify_max_ntiles(kv0.head_dim))
    return fail(VEGAS_ERR_UNSUPPORTED, "(gamma+1)*G = %d query rows exceeds this head_dim's limit",
                (gamma + 1) * G);
  if (G > 16) return fail(VEGAS_ERR_UNSUPPORTED, "group size %d (at most 16)", G);
  if ((long long)k_max + max_tail > vegas::kMaxSparseCluster * vegas::kMaxSparseRowsPerCta)
    return fail(VEGAS_ERR_UNSUPPORTED, "k_max + max_tail = %lld exceeds %d",
                (long long)k_max + max_tail, vegas::kMaxSparseCluster * vegas::kMaxSparseRowsPerCta);
  if ((long long)score_stride > 8ll * vegas::select_max_chunk())
    return fail(VEGAS_ERR_UNSUPPORTED, "score_stride %d exceeds %d", score_stride,
                8 * vegas::select_max_chunk());
  if (batch == 0) return VEGAS_OK;
  int dev = 0;
  {
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(VEGAS_ERR_UNSUPPORTED, "device ordinal %d", dev);
  }
  vegas_status_t st = device_info(nullptr, nullptr);
  if (st != VEGAS_OK) return st;
  const size_t need = vegas_verify_workspace_size(&kv0, batch, gamma);
  if (need > 0 && (!workspace || workspace_bytes < need))
    return fail(VEGAS_ERR_WORKSPACE_TOO_SMALL, "verify workspace %zu < %zu bytes",
                workspace_bytes, need);

  // ---- enqueue
  EventPool& pool = g_event_pool[dev];
  std::lock_guard<std::mutex> lock(pool.mu);
  const bool piped = select_stream != nullptr;
  if (piped) {
    while ((int)pool.ev.size() < 2 * num_layers) {
      cudaEvent_t e = nullptr;
      cudaError_t ce = cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
      if (ce != cudaSuccess) return cuda_fail(ce, "cudaEventCreateWithFlags");
      pool.ev.push_back(e);
    }
  }
  cudaStream_t main_s = static_cast<cudaStream_t>(stream);
  cudaStream_t side_s = static_cast<cudaStream_t>(select_stream);
  for (int l = 0; l < num_layers; ++l) {
    const vegas_layer_t& L = layers[l];
    st = vegas_verify_attn_capture(&L.kv, L.q_verify, L.out_verify, L.scores, score_stride,
                                   ctx_lens, batch, gamma, 0, gamma, softmax_scale, workspace,
                                   workspace_bytes, stream);
    if (st != VEGAS_OK) return st;
    if (piped) {
      cudaError_t ce = cudaEventRecord(pool.ev[2 * l], main_s);
      if (ce == cudaSuccess) ce = cudaStreamWaitEvent(side_s, pool.ev[2 * l], 0);
      if (ce != cudaSuccess) return cuda_fail(ce, "verify -> select ordering");
    }
    st = vegas_select_topk(L.scores, score_stride, ctx_lens, k_per_seq, L.idx, batch,
                           L.kv.num_kv_heads, k_max, piped ? select_stream : stream);
    if (st != VEGAS_OK) return st;
    if (piped) {
      cudaError_t ce = cudaEventRecord(pool.ev[2 * l + 1], side_s);
      if (ce != cudaSuccess) return cuda_fail(ce, "select completion event");
    }
  }
  for (int j = 0; j < gamma; ++j) {
    for (int l = 0; l < num_layers; ++l) {
      const vegas_layer_t& L = layers[l];
      if (piped && j == 0) {
        cudaError_t ce = cudaStreamWaitEvent(main_s, pool.ev[2 * l + 1], 0);
        if (ce != cudaSuccess) return cuda_fail(ce, "select -> draft ordering");
      }
      const size_t qoff = size_t(j) * batch * L.kv.num_q_heads * L.kv.head_dim * 2;
      st = vegas_sparse_decode_attn(
          &L.kv, static_cast<const uint8_t*>(L.q_draft) + qoff,
          static_cast<uint8_t*>(L.out_draft) + qoff, L.idx, k_max, k_per_seq, ctx_lens,
          tail_lens + size_t(j) * batch, max_tail, batch, softmax_scale, stream);
      if (st != VEGAS_OK) return st;
    }
  }
  if (piped && gamma == 0) {
    // no draft step joined the select stream back: wait for its last select
    cudaError_t ce = cudaStreamWaitEvent(main_s, pool.ev[2 * (num_layers - 1) + 1], 0);
    if (ce != cudaSuccess) return cuda_fail(ce, "select join");
  }
  return VEGAS_OK;
}

// =========================================================================
// Failure-detection check
// =========================================================================
VEGAS_API vegas_status_t vegas_check_bounded_wait(int limit_us, int* outcome, void* stream) {
  if (limit_us < 1 || limit_us > 1000000)
    return fail(VEGAS_ERR_INVALID_ARG, "limit_us %d outside [1, 1000000]", limit_us);
  int* err = nullptr;
  vegas_status_t st = device_info(&err, nullptr);
  if (st != VEGAS_OK) return st;
  cudaError_t e = vegas::launch_bounded_wait_check(1000ull * (unsigned long long)limit_us, err,
                                                   outcome, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "bounded-wait check launch");
  return VEGAS_OK;
}

// =========================================================================
// Status
// =========================================================================
VEGAS_API vegas_status_t vegas_read_device_status(void* stream) {
  int* err = nullptr;
  vegas_status_t st = device_info(&err, nullptr);
  if (st != VEGAS_OK) return st;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int word = 0;
  e = cudaMemcpyFromSymbol(&word, g_error_word, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "read error word");
  if (word != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "clear error word");
    return fail(static_cast<vegas_status_t>(word), "device reported %s",
                vegas_status_string(static_cast<vegas_status_t>(word)));
  }
  return VEGAS_OK;
}

VEGAS_API const char* vegas_status_string(vegas_status_t s) {
  switch (s) {
    case VEGAS_OK: return "VEGAS_OK";
    case VEGAS_ERR_INVALID_ARG: return "VEGAS_ERR_INVALID_ARG";
    case VEGAS_ERR_UNSUPPORTED: return "VEGAS_ERR_UNSUPPORTED";
    case VEGAS_ERR_WORKSPACE_TOO_SMALL: return "VEGAS_ERR_WORKSPACE_TOO_SMALL";
    case VEGAS_ERR_CUDA: return "VEGAS_ERR_CUDA";
    case VEGAS_ERR_DEVICE_FAULT: return "VEGAS_ERR_DEVICE_FAULT";
    case VEGAS_ERR_DEVICE_TIMEOUT: return "VEGAS_ERR_DEVICE_TIMEOUT";
  }
  return "VEGAS_ERR_UNKNOWN";
}

VEGAS_API const char* vegas_last_error_detail(void) { return g_detail; }

VEGAS_API int vegas_abi_version(void) { return VEGAS_ABI_VERSION; }
