/*
 * vegas.h - C ABI of the Vegas hot path on one GB300 (sm_103a).
 *
 * Method: "Vegas: Self-Speculative Decoding with Verification-Guided Sparse
 * Attention" (Yue, Xue, Huang), gist.science technical summary of paper
 * 2602.07223.  One decode iteration runs
 *   (1) full verify attention over the paged KV cache, capturing the
 *       pre-softmax logits of the two Collect-2-Query rows summed per KV head
 *       (§2 "Core mechanism", §2.A equation, §2.B "Collect-2-Query",
 *       §3 "Implementation": logits taken before softmax normalisation);
 *   (2) a per-(sequence, KV head) top-k over those summed logits (§2.A);
 *   (3) gamma sparse draft-decode attention steps over the selected positions
 *       plus a dense tail (§2, §3: PagedAttention with one token per page).
 *
 * Conventions shared by every entry point:
 *  - Every pointer named "device" is a CUDA device pointer owned by the caller.
 *    The library keeps no reference to it after the call returns.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and runs asynchronously.  No entry point synchronises the host
 *    except vegas_read_device_status.
 *  - Arguments are validated on the host before anything is launched; a bad
 *    argument returns a status and launches nothing.  vegas_last_error_detail()
 *    then describes it (per host thread).
 *  - Faults only visible on the device (a block-table entry outside
 *    [0, num_pages), a selected index outside the sequence, k_b > L_b, a
 *    bounded wait that ran out) are recorded in a per-device error word; the
 *    kernel clamps the access, skips the work and returns.  Nothing traps.
 *    vegas_read_device_status() returns and clears that word.
 *  - Workspaces are caller-allocated device memory of at least the size the
 *    matching *_workspace_size() reports, zero-filled once before their first
 *    use (e.g. cudaMemsetAsync).  Every call leaves the workspace's counters
 *    at zero again.  A workspace must not be shared by calls that may run
 *    concurrently.  A reported size of 0 means the call needs none (NULL is
 *    accepted).
 *  - The library allocates no device memory in these calls.
 *  - Kernels are launched with programmatic dependent launch: each may begin
 *    while the previous kernel of the stream drains, and waits for that
 *    kernel to complete (griddepcontrol.wait) before touching global memory.
 *    A caller kernel launched with the same attribute right after one of
 *    these calls must wait likewise before reading its outputs.
 */
#ifndef VEGAS_H_
#define VEGAS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define VEGAS_ABI_VERSION 1
#define VEGAS_PAGE_SIZE 16

typedef enum {
  VEGAS_OK = 0,
  VEGAS_ERR_INVALID_ARG = 1,         /* host-side argument check failed; nothing launched */
  VEGAS_ERR_UNSUPPORTED = 2,         /* valid but outside the shapes this library supports */
  VEGAS_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes below the *_workspace_size() value */
  VEGAS_ERR_CUDA = 4,                /* a CUDA runtime call failed (see detail string) */
  VEGAS_ERR_DEVICE_FAULT = 5,        /* a kernel met an out-of-range page, index or k */
  VEGAS_ERR_DEVICE_TIMEOUT = 6       /* a kernel's bounded wait ran out */
} vegas_status_t;

/*
 * Paged KV cache (vLLM-style paging, §3).  K and V are separate bf16 tensors
 * laid out [num_pages][num_kv_heads][page_size][head_dim], so one (page,
 * KV head) block of 16 tokens is contiguous.  Logical position i of sequence b
 * lives in physical page block_table[b * max_pages_per_seq + i / 16], slot
 * i % 16.  Query head h reads KV head h / (num_q_heads / num_kv_heads).
 */
typedef struct {
  const void* k_cache;          /* device, bf16, 16-byte aligned */
  const void* v_cache;          /* device, bf16, 16-byte aligned */
  const int32_t* block_table;   /* device, int32 [batch][max_pages_per_seq] */
  int32_t num_pages;
  int32_t page_size;            /* must be 16 */
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;             /* 64 or 128 */
  int32_t max_pages_per_seq;
} vegas_paged_kv_t;

/* ------------------------------------------------------------------------
 * (1) Verify attention with Collect-2-Query capture.
 *
 * For sequence b with committed prefix L_b = ctx_lens[b] and window row
 * t in [0, gamma] (the window's K/V already sit at positions L_b .. L_b+gamma),
 * query head h attends positions [0, L_b + t]:
 *   l_ti = (q_t^h . k_i) * softmax_scale,  o_t^h = sum_i softmax(l)_i v_i.
 * If scores != NULL, also writes, for every KV head g and i in [0, L_b),
 *   scores[(b * num_kv_heads + g) * score_stride + i]
 *     = sum_{t in {capture_row_a, capture_row_b}} sum_{h in group g} l_ti^(h)
 * (fp32; the §2.A objective restricted to the two Collect-2-Query rows,
 * rows 0 and gamma under this library's reading).  capture_row_a ==
 * capture_row_b captures one row once.  Entries at i >= L_b are not written.
 *
 *   q:   device bf16 [batch][gamma + 1][num_q_heads][head_dim], 16-byte aligned
 *   out: device bf16, same shape as q, 16-byte aligned
 *   ctx_lens: device int32 [batch]; needs L_b + gamma + 1 <= 16 * max_pages_per_seq
 *   score_stride >= max_b L_b when scores != NULL
 * Supported: head_dim in {64, 128}; (gamma + 1) * G <= 64 with G = Hq / Hkv;
 * gamma in [0, 15].
 * ---------------------------------------------------------------------- */
size_t vegas_verify_workspace_size(const vegas_paged_kv_t* kv, int batch, int gamma);

vegas_status_t vegas_verify_attn_capture(
    const vegas_paged_kv_t* kv, const void* q, void* out, float* scores,
    int score_stride, const int32_t* ctx_lens, int batch, int gamma,
    int capture_row_a, int capture_row_b, float softmax_scale,
    void* workspace, size_t workspace_bytes, void* stream);

/*
 * (1'') Verify attention capturing any set of window rows.  The same call as
 * vegas_verify_attn_capture, with the captured rows given as a bit mask
 * (bit t set: row t, 0 <= t <= gamma) instead of two row numbers:
 *   scores[(b * num_kv_heads + g) * score_stride + i]
 *     = sum_{t in mask} sum_{h in group g} l_ti^(h).
 * §2.B "Collect-2-Query" contrasts its two rows with collecting the logits of
 * every draft row; capture_row_mask = 2^(gamma+1) - 1 is that collect-all
 * variant.  Here every variant costs the same: the captured rows enter the
 * kernel as one summed query (two extra MMA columns), not as logits written
 * per row.  Needs 0 < capture_row_mask < 2^(gamma+1) when scores != NULL.
 */
vegas_status_t vegas_verify_attn_capture_rows(
    const vegas_paged_kv_t* kv, const void* q, void* out, float* scores,
    int score_stride, const int32_t* ctx_lens, int batch, int gamma,
    uint32_t capture_row_mask, float softmax_scale, void* workspace,
    size_t workspace_bytes, void* stream);

/*
 * (1-raw) The pages' capture, for comparison (§3 "Implementation": the verify
 * kernel writes raw pre-softmax logits, aggregated afterwards).  Verify
 * attention as vegas_verify_attn_capture without its fused capture, writing
 * instead every captured row's logit of every query head:
 *   raw[((b * R + r) * num_q_heads + h) * raw_stride + i] = l_ti^(h)
 * for i in [0, min(L_b, raw_stride)), where t is the r-th set bit of
 * capture_row_mask and R its popcount (device fp32).  Then
 * vegas_aggregate_raw_logits forms the same scores as the fused capture:
 *   scores[(b * num_kv_heads + g) * score_stride + i]
 *     = sum_{r < num_rows} sum_{h in group g} raw[...][i],  i < L_b,
 * summed in fp32 in (r, h) order; max_len >= max_b L_b sizes its grid.
 * Needs L_b <= raw_stride and L_b <= score_stride for the aggregate.
 */
vegas_status_t vegas_verify_attn_raw_logits(
    const vegas_paged_kv_t* kv, const void* q, void* out, float* raw, int raw_stride,
    const int32_t* ctx_lens, int batch, int gamma, uint32_t capture_row_mask,
    float softmax_scale, void* workspace, size_t workspace_bytes, void* stream);

vegas_status_t vegas_aggregate_raw_logits(
    const float* raw, int raw_stride, const int32_t* ctx_lens, int batch, int num_rows,
    int num_q_heads, int num_kv_heads, int max_len, float* scores, int score_stride,
    void* stream);

/*
 * (1') Verify attention that allocates nothing.  The paper has no counterpart:
 * this is a convenience for callers that cannot allocate device memory, for
 * instance a plugin whose host framework owns every device allocation through
 * its own pool, or a decode loop that must never call cudaMalloc because it
 * can synchronise the device.  Same arguments and results as
 * vegas_verify_attn_capture, without the workspace: the split-KV scratch lives
 * in a fixed 16 MiB array inside the library's device memory (every GPU that
 * loads the library holds it until exit).  Shapes whose
 * vegas_verify_workspace_size() exceeds vegas_verify_noalloc_max_scratch_bytes()
 * are rejected with VEGAS_ERR_WORKSPACE_TOO_SMALL.  The first call on a device
 * looks up the array's device address, so make it before any stream capture.
 * All calls share the array: each call clears its counters on `stream`, and
 * calls whose GPU work overlaps (other streams or host threads) race.
 */
size_t vegas_verify_noalloc_max_scratch_bytes(void);

vegas_status_t vegas_verify_attn_capture_noalloc(
    const vegas_paged_kv_t* kv, const void* q, void* out, float* scores,
    int score_stride, const int32_t* ctx_lens, int batch, int gamma,
    int capture_row_a, int capture_row_b, float softmax_scale, void* stream);

/* ------------------------------------------------------------------------
 * (2) Top-k select (§2.A argmax over |T| = k of the summed logits).
 *
 * For every (b, g): the k_b = k_per_seq[b] positions i in [0, L_b) of
 * largest scores[(b * num_kv_heads + g) * score_stride + i], ties going to
 * the lower position, written ascending to
 * out_idx[(b * num_kv_heads + g) * k_max + j], j < k_b; entries j >= k_b are
 * set to -1.  -0.0 ranks equal to +0.0.  NaN scores are outside the
 * contract (they rank lowest).  Needs 0 <= k_b <= min(L_b, k_max) and
 * L_b <= score_stride <= 262144.
 * ---------------------------------------------------------------------- */
vegas_status_t vegas_select_topk(
    const float* scores, int score_stride, const int32_t* ctx_lens,
    const int32_t* k_per_seq, int32_t* out_idx, int batch, int num_kv_heads,
    int k_max, void* stream);

/*
 * (2'') One T per sequence shared by every query head: the §2.A objective with
 * H = all query heads of the layer (the literal sum over heads) instead of the
 * G heads of one KV head.  Same arguments and layout as vegas_select_topk; the
 * score of position i is the fp32 sum, in KV-head order g = 0 .. Hkv-1, of
 * scores[(b * num_kv_heads + g) * score_stride + i], and the chosen positions
 * are written to the out_idx rows of every KV head of the sequence.
 */
vegas_status_t vegas_select_topk_shared(
    const float* scores, int score_stride, const int32_t* ctx_lens,
    const int32_t* k_per_seq, int32_t* out_idx, int batch, int num_kv_heads,
    int k_max, void* stream);

/*
 * (2') Query-agnostic selection: the sliding-window baseline that §1
 * "Problem" contrasts with verification-guided selection (cheap to select,
 * poorer drafts), with optional sink positions at the start of the prefix.
 * For every (b, g):
 *   T_b = [0, min(num_sink, L_b)) U [max(num_sink, L_b - window), L_b),
 * k_b = min(L_b, num_sink + window), written ascending in the layout of
 * vegas_select_topk (entries j >= k_b set to -1), and k_out[b] = k_b (device
 * int32 [batch]), ready for vegas_sparse_decode_attn.  Needs
 * k_max >= num_sink + window.  ctx_lens is device int32 [batch].
 */
vegas_status_t vegas_select_window(const int32_t* ctx_lens, int num_sink, int window,
                                   int32_t* k_out, int32_t* out_idx, int batch,
                                   int num_kv_heads, int k_max, void* stream);

/* ------------------------------------------------------------------------
 * (3) Sparse draft-decode attention, one draft step (§2, §3).
 *
 * For every b and query head h (KV head g = h / G), attends the positions
 *   idx[(b * num_kv_heads + g) * k_max + j] for j < k_per_seq[b]
 *   followed by tail_start[b] .. tail_start[b] + tail_len[b] - 1
 * with o = sum softmax((q . k_i) * softmax_scale) v_i.  idx entries are
 * logical positions (page size 1 semantics); each must lie inside the
 * block table's range.
 *   q, out: device bf16 [batch][num_q_heads][head_dim]
 *   max_tail >= max_b tail_len[b]; k_per_seq[b] + tail_len[b] >= 1.
 * Needs no workspace (the split softmax states merge on chip).
 * Supported: head_dim in {64, 128}, G <= 16, k_max + max_tail <= 32768
 * (up to 16 CTAs of 2048 entries each per (sequence, KV head)); larger
 * sets return VEGAS_ERR_UNSUPPORTED before anything is launched.
 * ---------------------------------------------------------------------- */
vegas_status_t vegas_sparse_decode_attn(
    const vegas_paged_kv_t* kv, const void* q, void* out, const int32_t* idx,
    int k_max, const int32_t* k_per_seq, const int32_t* tail_start,
    const int32_t* tail_len, int max_tail, int batch, float softmax_scale,
    void* stream);

/* ------------------------------------------------------------------------
 * (4) One decode iteration over a stack of layers (§2 "Core mechanism": each
 * layer's verify pass selects the entries its next draft phase attends; §4
 * puts the selection's cost at 5.9-9.4% of decode time).
 *
 * For every layer l in order: vegas_verify_attn_capture (capture rows 0 and
 * gamma) followed by vegas_select_topk on that layer's scores; then, for every
 * draft step j < gamma and every layer l, vegas_sparse_decode_attn over the
 * layer's indices and the tail
 *   [ctx_lens[b], ctx_lens[b] + tail_lens[j * batch + b]).
 * Layer-pipelined select: when select_stream is not NULL, select(l) runs on
 * select_stream and overlaps verify(l + 1) on `stream` (which does not depend
 * on it), and draft step 0 of layer l waits for select(l).  Every piece of
 * work is joined back into `stream`, so the call can be captured in a CUDA
 * graph on `stream`.  The cross-stream ordering uses events the library
 * creates once per device (2 per layer, grown to the largest layer count
 * seen): make the first call with a given layer count before any capture.
 * Calls are serialised per device on the host while they enqueue.
 *
 *   layers: host array of num_layers descriptors; every layer has the same
 *           batch, heads and head_dim (one model's stack); block tables may
 *           be shared.
 *   ctx_lens, k_per_seq: device int32 [batch] (L_b, k_b), as for verify/select
 *   tail_lens: device int32 [gamma][batch]; max_tail >= every entry
 *   workspace: verify workspace of vegas_verify_workspace_size(layer 0) bytes
 *              (layers run their verify one after another and share it)
 * Every argument is checked before anything is launched.
 * ---------------------------------------------------------------------- */
typedef struct {
  vegas_paged_kv_t kv;          /* this layer's caches */
  const void* q_verify;         /* device bf16 [batch][gamma + 1][Hq][d], 16-byte aligned */
  void* out_verify;             /* device bf16, same shape, 16-byte aligned */
  const void* q_draft;          /* device bf16 [gamma][batch][Hq][d], 16-byte aligned */
  void* out_draft;              /* device bf16, same shape */
  float* scores;                /* device fp32 [batch][Hkv][score_stride] */
  int32_t* idx;                 /* device int32 [batch][Hkv][k_max] */
} vegas_layer_t;

vegas_status_t vegas_decode_iteration(
    const vegas_layer_t* layers, int num_layers, const int32_t* ctx_lens,
    const int32_t* k_per_seq, const int32_t* tail_lens, int max_tail, int batch, int gamma,
    int score_stride, int k_max, float softmax_scale, void* workspace,
    size_t workspace_bytes, void* stream, void* select_stream);

/* ------------------------------------------------------------------------
 * Failure-detection check (the paper has no counterpart).
 *
 * Every wait of these kernels on an on-chip barrier (a TMA tile landing, an
 * MMA completing, a peer CTA's partial state) gives up after a time limit:
 * the kernel then records VEGAS_ERR_DEVICE_TIMEOUT in the device error word,
 * drains what it has in flight and returns, so a lost arrival cannot hang the
 * GPU.  This call shows that protocol end to end: it launches one CTA that
 * waits, with limit_us microseconds as its limit (1 .. 1000000), on a barrier
 * nothing ever arrives on (with nothing else in flight), records the timeout
 * and returns.  The next vegas_read_device_status() then returns
 * VEGAS_ERR_DEVICE_TIMEOUT and clears the word.  If outcome is not NULL
 * (device int32), it receives 0 when the wait ran out (1 if it completed).
 * ---------------------------------------------------------------------- */
vegas_status_t vegas_check_bounded_wait(int limit_us, int32_t* outcome, void* stream);

/* ------------------------------------------------------------------------
 * Status.
 * ---------------------------------------------------------------------- */
/* Synchronises `stream`, returns the current device's error word as a status
 * (VEGAS_OK when clear) and clears it. */
vegas_status_t vegas_read_device_status(void* stream);
const char* vegas_status_string(vegas_status_t status);
/* Human-readable detail of the last non-OK status returned on this host thread. */
const char* vegas_last_error_detail(void);
int vegas_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* VEGAS_H_ */
