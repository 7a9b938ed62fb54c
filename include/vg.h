/*
 * vg.h -- C ABI of the verification-guided self-speculative sparse attention
 * hot path on GB300 (sm_103a).
 *
 * Three calls make one decode step of a layer:
 *   vg_verify_attention        full-KV GQA attention of the k+1 verify rows,
 *                              capturing two logit rows (Collect-2-Query);
 *   vg_select_kv               sink + recent + top-k index list from them;
 *   vg_sparse_draft_attention  decode attention of one draft position over
 *                              the index list plus the dense tail.
 *
 * Sources (page title, section):
 *   Vegas: Self-Speculative Decoding with Verification-Guided Sparse
 *   Attention (arXiv 2602.07223) -- "The pith", "Core claim", "What carries
 *   the argument", Figure 1 and Figure 6 captions, Appendix A.
 *   A Sparse Glimpse of the Whole: Train-Free Self-Speculative Decoding
 *   (arXiv 2607.27735) -- "Core claim", "What carries the argument".
 *
 * Conventions shared by every call
 *   - Pointers are DEVICE pointers unless a comment says otherwise.  The
 *     caller owns and allocates all memory; the library never allocates,
 *     frees or synchronises.  Every call is asynchronous on `stream` and
 *     stream-ordered; per-sequence lengths live on the device and the host
 *     passes only upper bounds.
 *   - bf16 means IEEE bfloat16 stored as uint16.
 *   - Host-detectable problems return a status and launch nothing.
 *   - Device-detectable problems (page id out of range, index out of range,
 *     a length above the host bound, a pipeline wait that timed out) OR a
 *     VG_DEVERR_* bit into *error_flag (when error_flag is not NULL) and skip
 *     the offending load or sequence; nothing traps.
 *   - Workspaces: sized by the matching *_workspace_bytes() call for the same
 *     arguments on the same device (0 = none needed, the pointer may be
 *     NULL).  Calls that share a workspace must not overlap in time.  The
 *     verify and select workspaces need no initialisation: everything in
 *     them is written before it is read.  The sparse draft needs none.
 */
#ifndef VG_H_
#define VG_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum vg_status {
  VG_OK = 0,
  VG_ERR_INVALID_ARGUMENT = 1,   /* null pointer, negative size, inconsistent shape */
  VG_ERR_UNSUPPORTED = 2,        /* valid but outside the supported shapes        */
  VG_ERR_WORKSPACE_TOO_SMALL = 3,
  VG_ERR_LAUNCH = 4              /* a CUDA call failed; see cudaGetLastError()    */
} vg_status;

/* What vg_verify_attention writes to `capture`. */
enum {
  VG_CAPTURE_NONE = 0,
  /* float32 [batch][num_kv_heads][max_prefix]:
   *   G[b][h][j] = sum over the query heads q of KV head h, ascending, of
   *                (s[q][row 0][j] + s[q][row k][j]),
   *   accumulated in float32 as acc = pair(q0); acc = acc + pair(q1); ...   */
  VG_CAPTURE_GROUP_SUM = 1,
  /* float32 [batch][num_q_heads][2][max_prefix]: slot 0 = row 0 (first draft
   * token), slot 1 = row k (bonus token).  With n_rows == 1 both slots hold
   * row 0.                                                                  */
  VG_CAPTURE_ROWS = 2,
  /* Collect-All-Query (Vegas, Figure 6 and "Core claim": the costlier rule
   * that aggregates every verify row).  float32 [batch][num_kv_heads]
   * [max_prefix], same layout as VG_CAPTURE_GROUP_SUM:
   *   A[b][h][j] = sum over all n_rows rows and all query heads of KV head h
   *                of s[q][i][j].
   * Order: the g * n_rows (head, row) pairs are packed as [row 0 of each
   * head][row k of each head][rows 1..k-1, head-major within a row]; each
   * block of 32 consecutive pairs is reduced by a fixed butterfly, and the
   * blocks' sums are added in ascending block order.                       */
  VG_CAPTURE_ALL_SUM = 3,
  /* Every row, for attention-weight statistics (A Sparse Glimpse of the
   * Whole, "What carries the argument": rank by the post-softmax weights of
   * a window of verification queries; the window here is the n_rows block
   * rows).  float32, two consecutive arrays:
   *   logits [batch][num_q_heads][n_rows][max_prefix]: s[q][i][j] for the
   *          prefix positions j < L_b (the rest untouched);
   *   lse    [batch][num_q_heads][n_rows]: ln sum_{j <= L_b + i} exp(s[q][i][j]),
   *          the row's softmax normaliser over everything it attends.
   * Select on it with vg_select_kv_weights.                                */
  VG_CAPTURE_ALL_ROWS = 4
};

/* Bits OR-ed into *error_flag by the kernels. */
enum {
  VG_DEVERR_PAGE = 1,     /* page-table entry outside [0, num_pages)          */
  VG_DEVERR_INDEX = 2,    /* selected index outside [0, tail_start)           */
  VG_DEVERR_COUNT = 4,    /* selected count outside [0, cap]                  */
  VG_DEVERR_TIMEOUT = 8,  /* a pipeline wait outlasted its bound (see below)   */
  VG_DEVERR_LENGTH = 16   /* a device length exceeds its host-side bound      */
};

/* Paged KV cache.  Pages hold 16 consecutive positions of one sequence.
 *   k_pages, v_pages: bf16 [num_pages][num_kv_heads][page_size][head_dim];
 *                     base 16-byte aligned.  One (page, head) chunk is
 *                     contiguous (4 KB at head_dim 128).
 *   page_table:       int32 [batch][max_pages_per_seq]; logical page p of
 *                     sequence b is physical page page_table[b][p].  Entries
 *                     past a sequence's last page are never read.
 * Cache slots of the last page past a sequence's length may hold anything.  */
typedef struct vg_paged_kv {
  const void* k_pages;
  const void* v_pages;
  const int32_t* page_table;
  int32_t num_pages;
  int32_t page_size;           /* must be 16                    */
  int32_t max_pages_per_seq;
  int32_t num_kv_heads;
  int32_t head_dim;            /* 64 or 128                     */
} vg_paged_kv;

/* ---------------------------------------------------------------------------
 * Verification attention with Collect-2-Query capture.
 * Vegas, "Core claim" and Figure 6: one full-attention pass over the cache
 * verifies the k drafts plus the bonus position and writes only the
 * pre-softmax logit rows of the first draft token and of the bonus token.
 *
 *   q            bf16 [batch][n_rows][num_q_heads][head_dim], n_rows = k+1.
 *   prefix_lens  int32 [batch], 1 <= L_b <= max_prefix.  Verify row i of
 *                sequence b sits at position L_b + i and attends positions
 *                [0, L_b + i] (its own K/V must already be in the cache).
 *   softmax_scale  logits are softmax_scale * q.k (1/sqrt(head_dim) for the
 *                usual attention; 1 captures the raw qK^T).
 *   out          bf16 [batch][n_rows][num_q_heads][head_dim].
 *   capture      see VG_CAPTURE_*; only prefix positions j < L_b are
 *                written, the rest of each row is left untouched.  May be
 *                NULL with VG_CAPTURE_NONE.
 *   num_splits   0 = automatic; otherwise the number of KV-length splits
 *                (clamped to the number of 128-position tiles).  Results agree
 *                across split counts up to float32 rounding.  With more than
 *                one split, the call launches a second, small merge kernel
 *                (programmatic dependent launch) on the same stream.
 * Supported: head_dim 64/128, page_size 16, group g = num_q_heads /
 * num_kv_heads in [1, 8], g * n_rows <= 96, n_rows <= 16.
 * ------------------------------------------------------------------------- */
size_t vg_verify_workspace_bytes(int batch, int n_rows, int num_q_heads, int num_kv_heads,
                                 int head_dim, int max_prefix, int num_splits);

vg_status vg_verify_attention(const vg_paged_kv* kv, const void* q, const int32_t* prefix_lens,
                              int batch, int n_rows, int num_q_heads, int max_prefix,
                              float softmax_scale, void* out, int capture_mode, float* capture,
                              int num_splits, void* workspace, size_t workspace_bytes,
                              int32_t* error_flag, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Sparse verification, exact merged schedule.
 * SSV: Sparse Speculative Verification for Efficient LLM Inference, section
 * 4.2 and Figures 2, 4, 5: each verify row carries its own sparse selection,
 * and the blocks adjacent rows share are loaded once.
 *
 * Row i of sequence b attends the prefix positions of its selected blocks
 * plus the verify block causally:
 *   { j < L_b : j / 16 in blocks[b][i][0 .. block_counts[b][i]) }
 *     u [L_b, L_b + i].
 * The same selection serves every query head of the sequence.
 *
 *   blocks        int32 [batch][n_rows][max_blocks]: 16-position block
 *                 (logical page) numbers, each < ceil(L_b / 16); order and
 *                 duplicates do not matter.
 *   block_counts  int32 [batch][n_rows], 0 <= count <= max_blocks.
 *   q, prefix_lens, out, num_splits: as vg_verify_attention (no capture).
 *   workspace     vg_sparse_verify_workspace_bytes(); needs no
 *                 initialisation.
 *
 * Execution: a small kernel forms, per sequence, the ascending union of the
 * rows' blocks and the verify block's pages, with a row bit per page. The
 * verify kernel then streams that union once per KV head and masks each row
 * to its own blocks; a merge kernel follows when there is more than one
 * split.  Out-of-range blocks (VG_DEVERR_INDEX) and counts (VG_DEVERR_COUNT)
 * are flagged and skipped.
 * Supported: as vg_verify_attention, and max_pages_per_seq * 4 <= 200 KB.
 * ------------------------------------------------------------------------- */
size_t vg_sparse_verify_workspace_bytes(int batch, int n_rows, int num_q_heads, int num_kv_heads,
                                        int head_dim, int max_prefix, int max_blocks,
                                        int num_splits);

vg_status vg_sparse_verify_attention(const vg_paged_kv* kv, const void* q,
                                     const int32_t* prefix_lens, int batch, int n_rows,
                                     int num_q_heads, int max_prefix, float softmax_scale,
                                     const int32_t* blocks, const int32_t* block_counts,
                                     int max_blocks, void* out, int num_splits, void* workspace,
                                     size_t workspace_bytes, int32_t* error_flag,
                                     cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Verification-guided KV selection.
 * Vegas, "Core claim": combine the two captured rows across the query heads
 * and keep the top-k prefix positions.  A Sparse Glimpse of the Whole, "What
 * carries the argument": always keep sink and recent tokens; per-head index
 * variant.
 *
 * For each selection row (one per sequence, or one per KV head when
 * per_head != 0) the score of prefix position j is
 *   per_head == 0:  sum over KV heads h ascending of G[b][h][j]  (float32,
 *                   acc = G[0]; acc = acc + G[1]; ...),
 *   per_head != 0:  G[b][h][j],
 * where G is the capture itself (VG_CAPTURE_GROUP_SUM, or VG_CAPTURE_ALL_SUM,
 * which has the same layout) or is formed from VG_CAPTURE_ROWS in the order
 * documented above.  The result is
 *   [0, n_sink) u [L_b - n_recent, L_b) u (the top_k positions of
 *   [n_sink, L_b - n_recent) by score descending, lower position first on
 *   equal scores),
 * or all of [0, L_b) when L_b <= n_sink + n_recent + top_k.  -0.0 ranks as
 * +0.0.  Scores must not be NaN.
 *
 *   indices  int32 [batch][rows][cap], ascending, entries past the count = -1.
 *   counts   int32 [batch][rows].
 *   cap      >= min(max_prefix, n_sink + n_recent + top_k).
 *   kv, slots  optional (both NULL, or both given): slots int32
 *            [batch][rows][cap] receives, beside each kept position p, its
 *            cache slot page_table[b][p / 16] * 16 + p % 16 in kv's page
 *            pool (-1 past the count, and -1 with VG_DEVERR_PAGE where the
 *            page id is outside [0, num_pages)).  The translation is done
 *            once per selection, so that vg_sparse_draft_attention reaches a
 *            selected row in one dependent load.  kv->num_kv_heads must equal
 *            num_kv_heads and kv->max_pages_per_seq * 16 >= max_prefix.
 *   workspace  vg_select_workspace_bytes() bytes: room for the positions'
 *            score keys (one 4-byte key per prefix position and selection
 *            row); no initialisation needed.
 * The call launches one thread-block-cluster selection kernel on `stream`,
 * preceded by a score kernel that writes the keys to the workspace when the
 * cluster would have many capture loads per CTA (long prefixes, large
 * batches, raw-row and attention-weight captures); vg_select_launches() says
 * which.
 * Supported: max_prefix <= 262144, num_q_heads / num_kv_heads <= 8.
 * ------------------------------------------------------------------------- */
size_t vg_select_workspace_bytes(int batch, int num_kv_heads, int max_prefix, int per_head);

/* Kernels one vg_select_kv (capture_mode VG_CAPTURE_GROUP_SUM, _ALL_SUM or
 * _ROWS) or vg_select_kv_weights (VG_CAPTURE_ALL_ROWS) call launches for this
 * shape on the current device: 1 (the selection cluster forms the keys
 * itself) or 2 (a score kernel first).  The cluster size depends on how many
 * clusters the device holds at once, so the answer is device-specific.
 * Returns 0 for an invalid or unsupported shape.  Launches nothing. */
int vg_select_launches(int capture_mode, int batch, int num_kv_heads, int max_prefix,
                       int per_head);

vg_status vg_select_kv(const float* capture, int capture_mode, const int32_t* prefix_lens,
                       int batch, int num_q_heads, int num_kv_heads, int max_prefix, int top_k,
                       int n_sink, int n_recent, int per_head, int32_t* indices, int32_t* counts,
                       int cap, const vg_paged_kv* kv, int32_t* slots, void* workspace,
                       size_t workspace_bytes, int32_t* error_flag, cudaStream_t stream);

/* Weight-statistics variant of vg_select_kv (A Sparse Glimpse of the Whole,
 * "What carries the argument": rank positions by the attention weights of a
 * window of verification queries instead of two raw logit rows).  `capture`
 * is a VG_CAPTURE_ALL_ROWS capture of n_rows (<= 16) verify rows.  The score
 * of prefix position j is
 *   sum over the selection row's query heads q (ascending) and rows i
 *   (ascending) of expf(logits[q][i][j] - lse[q][i]),
 * i.e. the row-normalised post-softmax weights summed over the window (the
 * mean ranks identically); float32, fixed order.  Everything else --
 * candidates, sink/recent, ties, outputs, slots, workspace, errors -- is as
 * in vg_select_kv. */
vg_status vg_select_kv_weights(const float* capture, int n_rows, const int32_t* prefix_lens,
                               int batch, int num_q_heads, int num_kv_heads, int max_prefix,
                               int top_k, int n_sink, int n_recent, int per_head,
                               int32_t* indices, int32_t* counts, int cap,
                               const vg_paged_kv* kv, int32_t* slots, void* workspace,
                               size_t workspace_bytes, int32_t* error_flag, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Sparse draft attention.
 * Vegas, "Core claim" and Figure 1: while drafting, each draft token attends
 * only the selected KV entries; the positions produced since the selection
 * (the dense tail) are attended in full.
 *
 *   q           bf16 [batch][num_q_heads][head_dim], one draft position per
 *               sequence, at position cur_len[b] - 1.
 *   indices, counts  as written by vg_select_kv (per_head must match);
 *               every index must be < tail_start[b].
 *   slots       NULL, or the cache slots vg_select_kv wrote beside the
 *               indices (same shape): the K/V row of a selected entry is
 *               then read at its slot without a page-table lookup.  A slot
 *               whose offset within its page differs from its index's is
 *               flagged VG_DEVERR_INDEX and skipped.  Slots stay valid while
 *               the page-table entries of the selected positions do not
 *               change (new pages for the tail do not matter).
 *   tail_start  int32 [batch]: the prefix length the selection was made on.
 *   cur_len     int32 [batch]: query position + 1; tail = [tail_start,
 *               cur_len), 0 <= cur_len - tail_start <= max_tail.  The tail's
 *               rows are always reached through the page table.
 *   out         bf16 [batch][num_q_heads][head_dim]; zero when nothing is
 *               attended (count 0 and an empty tail).
 *   workspace   none needed: vg_sparse_draft_workspace_bytes() returns 0;
 *               the pointer and size are ignored (they may be NULL / 0).
 * One kernel: the attended list (selection, then tail) is processed in
 * chunks of 64 entries, cut into up to 16 segments, one CTA each; the
 * segments of a (sequence, KV head) form one thread-block cluster and their
 * fp32 records (m, l, O) are merged by the cluster's first CTA through
 * distributed shared memory, which writes `out`.
 * Supported: head_dim 64/128, g in [1, 8], cap + max_tail <= 65536.
 * ------------------------------------------------------------------------- */
size_t vg_sparse_draft_workspace_bytes(int batch, int num_q_heads, int num_kv_heads,
                                       int head_dim, int cap, int max_tail);

vg_status vg_sparse_draft_attention(const vg_paged_kv* kv, const void* q, const int32_t* indices,
                                    const int32_t* slots, const int32_t* counts, int per_head,
                                    int cap, const int32_t* tail_start, const int32_t* cur_len,
                                    int batch, int num_q_heads, int max_tail, float softmax_scale,
                                    void* out, void* workspace, size_t workspace_bytes,
                                    int32_t* error_flag, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Allocation-free verification attention.  The pages have no counterpart:
 * this entry point exists for callers that cannot allocate device memory --
 * for example an inference runtime that owns every byte of HBM through its
 * own pool and forbids libraries from calling cudaMalloc, or a decode loop
 * that must not call an allocator because cudaMalloc/cudaFree can
 * synchronise the device.  It computes exactly what vg_verify_attention
 * computes (same arguments minus the workspace) and allocates nothing.
 *
 * Its split-K scratch is one fixed device array of
 * vg_verify_noalloc_scratch_bytes() bytes (16 MiB), held by every GPU that
 * loads the library until the process exits.  Shapes needing more scratch
 * than that (vg_verify_workspace_bytes() above it) are rejected with
 * VG_ERR_WORKSPACE_TOO_SMALL before anything is launched; use
 * vg_verify_attention with a caller workspace for those.
 *
 *   - The scratch array belongs to the CURRENT device: call with the
 *     device of `stream` current (a stream of another device is rejected
 *     with VG_ERR_INVALID_ARGUMENT before anything is launched).
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make
 *     that first call before any stream capture.
 *   - Every call shares the one array, which keeps the last call's contents
 *     (nothing in it needs to start at zero); two calls that overlap on the
 *     GPU (different streams, no ordering between them) race on it.
 *   - No cudaMalloc, cudaFree or allocating library routine is called.
 * ------------------------------------------------------------------------- */
size_t vg_verify_noalloc_scratch_bytes(void);

vg_status vg_verify_attention_noalloc(const vg_paged_kv* kv, const void* q,
                                      const int32_t* prefix_lens, int batch, int n_rows,
                                      int num_q_heads, int max_prefix, float softmax_scale,
                                      void* out, int capture_mode, float* capture,
                                      int num_splits, int32_t* error_flag, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Failure detection: the bound on pipeline waits (host).
 * Every wait of a kernel on a copy, a tensor-core operation or another warp
 * is bounded.  A wait longer than `limit_ns` ORs VG_DEVERR_TIMEOUT into
 * *error_flag and goes on waiting, up to 1 s in all; so a short bound
 * reports slow waits without abandoning work in flight, and the call's
 * results are still complete.  A wait that outlasts 1 s is abandoned: the
 * kernel stops issuing work, waits (again at most 1 s) for the copies and
 * tensor-core operations it already issued, and returns with the flag set;
 * its outputs are then undefined.
 *   limit_ns  0 restores the default (1 s).  Takes effect for calls made
 *             after it returns, on every device; not synchronised with calls
 *             made concurrently from other host threads.
 * ------------------------------------------------------------------------- */
vg_status vg_set_wait_limit_ns(uint64_t limit_ns);

/* Static string for a status code (host). */
const char* vg_status_string(vg_status status);

/* Library version, e.g. "0.1.0" (host). */
const char* vg_version(void);

#ifdef __cplusplus
}
#endif
#endif /* VG_H_ */
