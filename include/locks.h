/*
 * locks.h — C ABI of the LOCKS decode-step library (liblocks.so), GB300 / sm_103a.
 *
 * LOCKS ("Page-Local Compact Key Summaries for Efficient Long-Context
 * Decoding", arXiv:2607.24555) keeps, for every full page of a paged KV cache,
 * a resident rank-r spectral summary of the page's keys: a basis V_j (d x r)
 * and per-token coefficients c_i (the rows of C_j = U_r Sigma_r, P x r).  Each
 * decode step projects every query onto every page basis, rebuilds the
 * within-page logits, estimates each page's attention mass by log-sum-exp,
 * averages the per-head mass shares over each GQA group, keeps the top pages
 * within a token budget without reading any candidate key or value, and then
 * runs exact attention over the selected pages plus the open tail.
 *
 * Passages defining the operations (page title, section):
 *   [expl] gist.science explainer, "Technische Samenvatting" §2 Methodologie:
 *          "Kernmechanisme" (summary = top-r eigenvectors of the page's keys
 *          plus per-token coefficients, built when a page is finalised),
 *          "Reconstructie en Selectie" (the equation for s_hat_j(q); ranking by
 *          estimated mass; no candidate key or value is read),
 *          "Group-Shared Selection (GSA)" (average of the estimated mass share
 *          over the query heads of a group -> one table per KV head),
 *          "Implementatie" (whole decode step inside CUDA graphs; summary
 *          construction off the critical path).
 *   [abs]  LOCKS abstract (insight.aitobox.com page, English paragraphs).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All pointers in the structs and arguments are DEVICE pointers unless
 *    stated otherwise.  The query, output and lse buffers (q, out, lse) may
 *    instead be page-locked host memory that the device can address
 *    (cudaHostAlloc / cudaHostRegister with unified addressing): the kernels
 *    then read the query and write the results in place over the CPU-GPU
 *    link, with no separate copy.  The caller owns every buffer and the stream; the
 *    library allocates nothing, frees nothing and never synchronises the
 *    stream (except locks_get_device_error, which reads back one word).
 *  - Element types: keys, values, queries, outputs and summaries are bf16
 *    (raw 16-bit patterns), lengths and indices int32, scores float32.
 *  - Supported sizes: head_dim d = 128, page_size P = 64 or 16 (the
 *    explainer's §2 "Kernmechanisme" gives a page size of 16), group size
 *    G = num_q_heads / num_kv_heads in 1..16, summary rank r even in 2..16
 *    (and r <= P).  Other values return LOCKS_ERR_UNSUPPORTED.
 *  - Query head hq belongs to KV head hq / G (standard GQA grouping).
 *  - Lengths (seq_lens, n_summarized) are read on the device, so a call can be
 *    captured once in a CUDA graph and replayed while the cache grows; all
 *    launch shapes depend only on the host-side struct fields.
 *  - Every call validates its host-side arguments before launching anything;
 *    on error nothing is launched.  Device-side range violations (a block
 *    table entry outside [0, pages_total), a selected page outside the
 *    sequence) skip the offending work and set a bit in the workspace's error
 *    word; read it with locks_get_device_error.  No call traps or aborts.
 *  - Scale: logits are q.k * scale with scale = 1/sqrt(d) when params.scale
 *    is 0.  Natural logarithms throughout.
 *  - No C++ exception crosses this interface.
 */
#ifndef LOCKS_H_
#define LOCKS_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define LOCKS_API __attribute__((visibility("default")))
#else
#define LOCKS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LOCKS_OK = 0,
  LOCKS_ERR_INVALID_ARG = 1,   /* null pointer, negative size, inconsistent shapes */
  LOCKS_ERR_UNSUPPORTED = 2,   /* a size the library does not implement (d, P, G, r) */
  LOCKS_ERR_CUDA = 3,          /* a CUDA runtime call or kernel launch failed */
  LOCKS_ERR_WORKSPACE = 4,     /* workspace missing, too small or misaligned */
  LOCKS_ERR_DEVICE = 5         /* returned by locks_get_device_error when a bit is set */
} locks_status_t;

/* Bits of the device error word. */
#define LOCKS_DEVERR_BLOCK_TABLE 0x1  /* block_table entry outside [0, pages_total) */
#define LOCKS_DEVERR_SEL_PAGE    0x2  /* selected page outside [0, n_summarized) */
#define LOCKS_DEVERR_LENGTHS     0x4  /* seq_len > max_pages * P or n_summarized > seq_len / P (clamped) */
#define LOCKS_DEVERR_PAGE_ID     0x8  /* builder page id outside [0, pages_total) */
#define LOCKS_DEVERR_TIMEOUT     0x10 /* a bounded wait on a TMA copy gave up (should never happen) */

#define LOCKS_DTYPE_BF16 0
#define LOCKS_DTYPE_F32 1
#define LOCKS_DTYPE_Q4 2
#define LOCKS_DTYPE_BF16_PACKED 3

/* Bytes of one page-head of a LOCKS_DTYPE_Q4 summary at rank r and page size
 * P (head_dim 128): 64r basis + 128 centroid + P r coefficients + 4(2r+1)
 * scales, rounded up to 16.  LOCKS_Q4_PAGE_HEAD_BYTES is the P = 64 case. */
#define LOCKS_Q4_BLOCK_BYTES(r, P) ((((72 * (r)) + ((P) * (r)) + 132) + 15) / 16 * 16)
#define LOCKS_Q4_PAGE_HEAD_BYTES(r) LOCKS_Q4_BLOCK_BYTES(r, 64)

/* Paged KV cache.  K and V pools hold whole pages for all KV heads:
 *   k_pool, v_pool  bf16 [pages_total][num_kv_heads][page_size][head_dim]
 *                   (one page-head = P x d contiguous, 16 KiB at P=64, d=128,
 *                   4 KiB at P=16;
 *                   base 16-byte aligned)
 *   block_table     int32 [batch][max_pages]: physical page of logical page j
 *                   of sequence b; entries past the sequence are not read
 *   seq_lens        int32 [batch]: tokens in the cache, current token included
 *   n_summarized    int32 [batch]: leading full pages whose summaries are
 *                   valid; pages from n_summarized on (full or partial) form
 *                   the open tail and are always attended.  May be NULL for
 *                   calls that do not select (dense decode, builder). */
typedef struct locks_cache {
  const void* k_pool;
  const void* v_pool;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const int32_t* n_summarized;
  int32_t batch;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t page_size;
  int32_t pages_total;
  int32_t max_pages;
} locks_cache_t;

/* Resident page summaries, indexed by PHYSICAL page like the pools:
 *   basis_t  [pages_total][num_kv_heads][rank][head_dim]: row j is the j-th
 *            basis vector (V_j transposed), descending singular value
 *   coeffs   [pages_total][num_kv_heads][page_size][rank]: row i is c_i
 *   dtype    LOCKS_DTYPE_BF16 for everything that reads summaries;
 *            LOCKS_DTYPE_F32 is accepted by locks_build_summaries only (a
 *            full-precision copy for validation);
 *            LOCKS_DTYPE_BF16_PACKED: the same bf16 values in one block per
 *            page-head, basis_t pointing to [pages_total][num_kv_heads]
 *            [rank * head_dim + page_size * rank]: the rank basis rows (as
 *            basis_t above) followed by the page_size x rank coefficients
 *            (as coeffs above); coeffs is unused.  The scan fetches a page's
 *            blocks for several KV heads with one copy instead of two, which
 *            makes it the faster bf16 layout;
 *            LOCKS_DTYPE_Q4: the quantised, centred format of the explainer's
 *            §2 "Kernmechanisme", Kwantisatie (int4 basis, int8 coefficients and centroid),
 *            rank 2..8.  Then basis_t points to one block of
 *            LOCKS_Q4_BLOCK_BYTES(rank, page_size) bytes per page-head,
 *            [pages_total][num_kv_heads][bytes], and coeffs is unused:
 *              byte 0       basis: row j (j < rank) at 64 j, 16 little-endian
 *                           32-bit words; word m (m = 0..15) holds elements
 *                           8m .. 8m+7 of the row, element 8m+i in bits
 *                           4(i/2) + 16(i%2) .. +3, as the code + 8 (codes in
 *                           [-7, 7]), and sits at word position 4(m%4) + m/4
 *                           of the row
 *              byte 64r     centroid mu: 128 bytes, code + 128 (codes in
 *                           [-127, 127])
 *              byte 64r+128 coefficients: P r bytes, code + 128; the code of
 *                           token i, column j at byte
 *                           (((i%8) (r/2) + j/2) (P/8) + i/8) 2 + j%2
 *              byte 64r+128+P r  float32 scales: for each column pair
 *                           t = 0 .. r/2-1 the four values s_v[2t],
 *                           s_v[2t+1], s_c[2t], s_c[2t+1]; then s_mu
 *            (the orders put the pieces one GPU lane needs side by side).
 *            The summary stands for V_j = s_v[j] * code, c_i[j] = s_c[j] *
 *            code, mu = s_mu * code, and the page's keys are approximated
 *            by mu + sum_j c_i[j] V_j (centred). */
typedef struct locks_summary {
  void* basis_t;
  void* coeffs;
  int32_t rank;
  int32_t dtype;
} locks_summary_t;

/* Decode parameters.  k_max = min(budget_tokens / page_size, max_pages) pages
 * are selected per (sequence, KV head), fewer when fewer pages are
 * summarised. */
typedef struct locks_params {
  int32_t num_q_heads;
  int32_t budget_tokens;
  float scale;     /* 0 -> 1/sqrt(head_dim) */
  int32_t flags;   /* 0, LOCKS_FLAG_UNFUSED or LOCKS_FLAG_FUSED; other bits are reserved and must be 0 */
} locks_params_t;

/* locks_decode_step runs as three kernels (summary scan, top-k, attention).
 * With LOCKS_FLAG_FUSED it runs as two when page_size is 64, k_max <= 32 and
 * max_pages <= 128 x (the largest thread-block cluster, 16 CTAs): the scan,
 * then one attention kernel whose clusters compute the group-shared top-k
 * themselves.  Both forms select the same pages; on GB300 the three-kernel
 * form is the faster one at every measured shape (1 to 256 problems).
 * LOCKS_FLAG_UNFUSED asks for the three-kernel form explicitly.  Setting both
 * is an error. */
#define LOCKS_FLAG_UNFUSED 0x1
#define LOCKS_FLAG_FUSED 0x2

/* Human-readable name of a status code (static string). */
LOCKS_API const char* locks_status_string(locks_status_t status);

/* Bytes of workspace needed by locks_select, locks_sparse_attend,
 * locks_decode_step and locks_dense_decode for these shapes (the maximum over
 * the four).  `summary` may be NULL when only attention calls are made.  The
 * workspace must be 256-byte aligned and zeroed once (locks_workspace_init)
 * before its first use; every call leaves its counters at zero again.  One
 * workspace must not be used by two calls that overlap on the GPU. */
LOCKS_API locks_status_t locks_workspace_size(const locks_cache_t* cache, const locks_summary_t* summary,
                                    const locks_params_t* params, size_t* bytes);

/* Zero `bytes` of workspace on `stream` (cudaMemsetAsync; capturable). */
LOCKS_API locks_status_t locks_workspace_init(void* ws, size_t bytes, void* stream);

/* Build summaries of n physical pages for every KV head ([expl] §2
 * "Kernmechanisme": when a page is finalised its keys get a small
 * eigendecomposition; the top-r eigenvectors and the per-token coefficients
 * are kept).  For each listed page-head K (P x d): the top-r eigenvectors U_r
 * of the Gram matrix K K^T (subspace iteration + Rayleigh-Ritz, fp32), then
 * V_r = orthonormalised K^T U_r and C = K V_r (= U_r Sigma_r).  Columns with
 * singular value <= 1e-6 sigma_1 are zero.  page_ids: device int32 [n];
 * an id outside [0, pages_total) is skipped and, when `ws` is given, sets
 * LOCKS_DEVERR_PAGE_ID.  `ws` may be NULL (then such errors are silent).
 * Reads k_pool only; block_table, seq_lens and v_pool are not used.
 * Capturable. */
LOCKS_API locks_status_t locks_build_summaries(const locks_cache_t* cache, locks_summary_t* summary,
                                     const int32_t* page_ids, int32_t n,
                                     void* ws, size_t ws_bytes, void* stream);

/* Page selection ([expl] §2 "Reconstructie en Selectie" and "GSA"; [abs]):
 * for every (b, KV head h) and every summarised page j < n_summarized[b] and
 * every query head g of the group
 *   s_hat[g][j] = ln sum_{i<P} exp( scale * (V_j^T q_g) . c_i )
 * then Z_g = ln sum_j exp(s_hat[g][j]),
 *   sigma_j = ln( (1/G) sum_g exp(s_hat[g][j] - Z_g) ),
 * and the k = min(k_max, n_summarized[b]) pages of largest sigma (ties to the
 * lower page) are written, ascending, to
 *   sel_pages  int32 [batch][num_kv_heads][k_max] (logical page numbers;
 *              slots past sel_count are not written)
 *   sel_count  int32 [batch][num_kv_heads]
 *   page_lse   optional float32 [batch][num_q_heads][max_pages]: s_hat for
 *              j < n_summarized[b] (other slots untouched); NULL to skip.
 * q: bf16 [batch][num_q_heads][head_dim].  Reads no key or value. */
LOCKS_API locks_status_t locks_select(const locks_cache_t* cache, const locks_summary_t* summary,
                            const locks_params_t* params, const void* q,
                            int32_t* sel_pages, int32_t* sel_count, float* page_lse,
                            void* ws, size_t ws_bytes, void* stream);

/* The summary scan alone ([expl] §2 "Reconstructie en Selectie", the
 * equation for s_hat_j(q)): page_lse[b][hq][j] = s_hat for every summarised
 * page j < n_summarized[b] (float32 [batch][num_q_heads][max_pages]; other
 * slots untouched), reading only the resident summaries.  This is the first
 * kernel of locks_select, exposed for callers with their own ranking. */
LOCKS_API locks_status_t locks_page_scores(const locks_cache_t* cache, const locks_summary_t* summary,
                                           const locks_params_t* params, const void* q, float* page_lse,
                                           void* ws, size_t ws_bytes, void* stream);

/* Exact attention over the selected pages plus the open tail (pages
 * n_summarized[b] .. ceil(seq_len/P)-1, the last one cut at seq_len):
 *   out[b][hq][:] = sum_t softmax_t(scale * q.k_t) v_t   (bf16 [batch][num_q_heads][head_dim])
 *   lse[b][hq]    = ln sum_t exp(scale * q.k_t)          (float32, optional)
 * sel_pages / sel_count as written by locks_select (stride k_max). */
LOCKS_API locks_status_t locks_sparse_attend(const locks_cache_t* cache, const locks_params_t* params,
                                   const void* q, const int32_t* sel_pages,
                                   const int32_t* sel_count, void* out, float* lse,
                                   void* ws, size_t ws_bytes, void* stream);

/* locks_select followed by locks_sparse_attend in one call (no host work
 * between the launches, programmatic dependent launch between kernels).
 * sel_pages / sel_count may be NULL (then kept in the workspace); when given
 * they receive the page list as locks_select writes it.  This is the whole
 * decode step; capture it in a CUDA graph for replay.  With LOCKS_FLAG_FUSED,
 * where the shapes allow, the top-k runs inside the attention kernel: each
 * sequence's thread-block cluster scores its pages, exchanges its best
 * candidates through distributed shared memory and attends to the pages it
 * selected, and the K/V of the open tail is loaded while the scan is still
 * running. */
LOCKS_API locks_status_t locks_decode_step(const locks_cache_t* cache, const locks_summary_t* summary,
                                 const locks_params_t* params, const void* q, void* out,
                                 float* lse, int32_t* sel_pages, int32_t* sel_count,
                                 void* ws, size_t ws_bytes, void* stream);

/* Number of kernels one locks_decode_step launches for these shapes and
 * flags: 2 (the scan, then attention with the top-k inside its clusters) or 3
 * (scan, top-k, attention); see LOCKS_FLAG_FUSED.  Host only; launches
 * nothing. */
LOCKS_API locks_status_t locks_decode_step_launches(const locks_cache_t* cache, const locks_summary_t* summary,
                                                    const locks_params_t* params, int32_t* launches);

/* Dense paged decode over every token of every sequence (the in-library
 * baseline the sparse step is measured against).  Same outputs as
 * locks_sparse_attend.  n_summarized is not read. */
LOCKS_API locks_status_t locks_dense_decode(const locks_cache_t* cache, const locks_params_t* params,
                                  const void* q, void* out, float* lse,
                                  void* ws, size_t ws_bytes, void* stream);

/* Exact page log-sum-exp that reads every key (the "read-every-key exact-LSE
 * oracle" of [abs]): page_lse[b][hq][j] = ln sum_{t in page j} exp(scale*q.k_t)
 * for every page j < ceil(seq_len/P) (cut at seq_len); other slots untouched.
 * A measurement helper for attention-mass recall, not part of the step. */
LOCKS_API locks_status_t locks_exact_page_lse(const locks_cache_t* cache, const locks_params_t* params,
                                    const void* q, float* page_lse, void* stream);

/* Capacity, in bytes, of the library's own static device workspace used by
 * locks_decode_step_static. */
#define LOCKS_STATIC_WS_BYTES ((size_t)8 << 20)

/* locks_decode_step for callers that cannot allocate device memory: hosts
 * that keep every byte of the GPU in their own pool and forbid outside
 * allocations, or thin C callers with no way to keep a workspace alive
 * between calls.  The paper has no counterpart; this is a convenience of
 * this library.
 *
 * Same arguments and results as locks_decode_step, minus the workspace: the
 * step runs in a fixed array of LOCKS_STATIC_WS_BYTES (8 MiB) that the
 * library holds in every CUDA context it is loaded in, until the context
 * ends.  Nothing is allocated or freed: no cudaMalloc, cudaFree or
 * allocating library routine is called.
 *   - Each call made outside stream capture looks up the array's device
 *     address in the current context (with cudaGetSymbolAddress); a call
 *     being captured reuses the address of the last uncaptured call on that
 *     device, and returns LOCKS_ERR_CUDA if there was none.  So make one
 *     uncaptured call on a device before capturing calls there, and again
 *     after cudaDeviceReset (which ends the context and its array).
 *   - Each call first zeroes the part of the array these shapes use (one
 *     cudaMemsetAsync on `stream`), so it does not depend on what an earlier
 *     call left there.
 *   - Every call on a device shares the one array: calls that overlap on the
 *     GPU (different streams, or different threads without ordering) race
 *     and give wrong results.  Order them on one stream.
 *   - Shapes whose workspace (locks_workspace_size) exceeds
 *     LOCKS_STATIC_WS_BYTES return LOCKS_ERR_WORKSPACE before any GPU work;
 *     use locks_decode_step with a caller-owned workspace for those.
 *   - device_error: optional device int32; receives this call's
 *     LOCKS_DEVERR_* bits (0 when none).  NULL to skip. */
LOCKS_API locks_status_t locks_decode_step_static(const locks_cache_t* cache, const locks_summary_t* summary,
                                                  const locks_params_t* params, const void* q, void* out,
                                                  float* lse, int32_t* sel_pages, int32_t* sel_count,
                                                  int32_t* device_error, void* stream);

/* Read (and clear) the workspace's device error word.  Synchronises `stream`.
 * *code receives the LOCKS_DEVERR_* bits; returns LOCKS_ERR_DEVICE when any
 * bit was set, LOCKS_OK otherwise.  Not capturable. */
LOCKS_API locks_status_t locks_get_device_error(void* ws, int32_t* code, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LOCKS_H_ */
