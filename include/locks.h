/*
 * locks.h - C ABI of the LOCKS decode-step library for GB300 (sm_103a).
 *
 * LOCKS ("page-local compact key summaries") keeps, for every 16-token page
 * of a paged bf16 K/V cache and every kv head, a small resident summary of
 * the page's keys, and at each decode step reads only those summaries to
 * choose the pages that receive full attention. Source pages:
 *   [post]    "LOCKS: per-page SVD cuts KV cache reads 10x at 1M context"
 *             (wps.hkprog.org), sections "How LOCKS works" and "Code"; for
 *             the ablations also "Why shared-basis sparse attention is
 *             structurally broken" and "Caveats".
 *   [summary] gist.science technical summary of arXiv 2607.24555, section 2
 *             "Method" (2.1 page-local spectral decomposition, 2.2
 *             reconstruction and selection, 2.3 group-shared selection,
 *             2.4 implementation); for the ablations also section 1 (problem
 *             statement: exact selection reads every key) and section 3
 *             (contributions: Proposition 1, the read-all-keys selector).
 *
 * Conventions shared by every call
 * --------------------------------
 * - Pointers named *_cache, q, scores, selected, out, lse, workspace and the
 *   summary arrays are DEVICE pointers (16-byte aligned; scales 8-byte).
 *   dims is a HOST pointer. The caller owns every buffer; the library
 *   allocates nothing and keeps no state besides cached device attributes.
 * - stream is a cudaStream_t passed as void* (NULL = the legacy default
 *   stream). Every call is asynchronous on that stream, performs no host
 *   synchronisation and no allocation, and so may be captured in a CUDA graph.
 * - Return value: LOCKS_OK, or a negative LOCKS_ERR_* code. Argument errors
 *   are detected on the host before anything is launched. LOCKS_ERR_CUDA means
 *   a launch failed (cudaGetLastError was not cudaSuccess). Errors that can
 *   only be seen on the device (a bounded wait that ran out) are recorded in
 *   the device status word at the start of the workspace; read it with
 *   locks_get_device_status. The standalone calls accept workspace = NULL
 *   (then device-side errors are not recorded); locks_decode_step needs
 *   locks_workspace_size bytes. Page ids read on the device are range-checked
 *   (LOCKS_ERR_BAD_INDEX) so a bad table cannot make a kernel read outside
 *   the caller's buffers.
 * - Fixed sizes: head_dim 128, page_size 16, rank 8. num_kv_heads must be 1,
 *   2, 4 or 8 and num_q_heads / num_kv_heads (the GQA group g) at most 16.
 *   Other values return LOCKS_ERR_UNSUPPORTED.
 * - Query head h attends through kv head h / g.
 *
 * Memory layouts
 * --------------
 *   k_cache, v_cache  bf16 bits [num_phys_pages][num_kv_heads][16][128]
 *   q                 fp32 [batch][num_q_heads][128]
 *   page_table        int32 [batch][max_pages_per_seq]: logical -> physical page
 *   seq_pages         int32 [batch]: full (summarised) pages of each sequence,
 *                     0 <= seq_pages[b] <= max_pages_per_seq
 *   scores            fp32 [batch][num_q_heads][max_pages_per_seq]
 *   lse_partials      fp32 pairs, locks_lse_partials_size bytes: (max, sum exp(score -
 *                     max)) of each sequence's scores per query head, split by the
 *                     scoring launch's CTAs and warps (an internal layout, written by
 *                     locks_score_pages and read by the selection calls for the same
 *                     dims on the same device); optional
 *   selected          int32 [batch][num_kv_heads][k_cap], ascending logical
 *                     page ids, k_cap = locks_k_cap(dims, budget_tokens)
 *   n_selected        int32 [batch][num_kv_heads]
 *   out               bf16 bits [batch][num_q_heads][128]
 *   lse               fp32 [batch][num_q_heads] (natural log), may be NULL
 *
 * Summary layout (one "unit" = one (physical page, kv head); 776 bytes)
 *   mu     int8  [num_phys_pages][num_kv_heads][128]
 *   basis  uint8 [num_phys_pages][num_kv_heads][512]  (int4 codes)
 *   coef   int8  [num_phys_pages][num_kv_heads][128]
 *   scales fp16 bits [num_phys_pages][num_kv_heads][4] = absmax scales of
 *          mu, basis, coef, then 0
 * Value = code * scale. Codes are symmetric: int8 in [-127, 127], int4 (two's
 * complement nibble) in [-7, 7]. Inside a unit, elements sit in the order the
 * scoring kernel's tensor-core fragments read them:
 *   mu[d]       at byte 32*t + 4*s + 2*h + e
 *   basis[d][r] in byte 64*r + 16*t + 4*(s/2) + p/2, nibble p%2 (0 = low 4 bits),
 *               p = 2*(s%2) + h + 4*e
 *   coef[i][r]  at byte 4*(4*(i%8) + r/2) + 2*(i/8) + r%2
 * where for a head dimension d: s = d/16, w = d%16, h = w/8, t = (w%8)/2,
 * e = w%2; i is the token (0..15) and r the rank (0..7).
 */
#ifndef LOCKS_H
#define LOCKS_H

#include <stddef.h>
#include <stdint.h>

#if defined(LOCKS_BUILD) && defined(__GNUC__)
#define LOCKS_API __attribute__((visibility("default")))
#else
#define LOCKS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define LOCKS_HEAD_DIM 128
#define LOCKS_PAGE_SIZE 16
#define LOCKS_MAX_TAIL_PAGES 4  /* pages without a summary that one tail may span */
#define LOCKS_RANK 8
#define LOCKS_MAX_GROUP 16
#define LOCKS_UNIT_BYTES 776

enum {
    LOCKS_OK = 0,
    LOCKS_ERR_INVALID_ARG = -1,        /* null pointer, negative or inconsistent size */
    LOCKS_ERR_UNSUPPORTED = -2,        /* head_dim/page/rank/heads outside what is built */
    LOCKS_ERR_WORKSPACE_TOO_SMALL = -3,
    LOCKS_ERR_CUDA = -4,               /* a CUDA runtime call or launch failed */
    LOCKS_ERR_TIMEOUT = -5,            /* device: a bounded wait ran out (status word) */
    LOCKS_ERR_BAD_INDEX = -6,          /* device: a page id or page-table entry out of range;
                                          the unit was skipped or read from page 0 instead */
};

typedef struct {
    int32_t batch;              /* B: sequences (requests) */
    int32_t num_q_heads;        /* Hq */
    int32_t num_kv_heads;       /* Hkv; g = Hq / Hkv */
    int32_t head_dim;           /* must be 128 */
    int32_t page_size;          /* must be 16 */
    int32_t rank;               /* must be 8 */
    int32_t max_pages_per_seq;  /* row stride of page_table and scores */
    int32_t num_phys_pages;     /* pages in the K/V pool and in the summary arrays */
} locks_dims_t;

typedef struct {
    int8_t* mu;         /* [num_phys_pages][Hkv][128]  device */
    uint8_t* basis;     /* [num_phys_pages][Hkv][512]  device */
    int8_t* coef;       /* [num_phys_pages][Hkv][128]  device */
    uint16_t* scales;   /* [num_phys_pages][Hkv][4]    device, fp16 bits */
} locks_summaries_t;

/* Library version (major * 10000 + minor * 100 + patch). */
LOCKS_API int locks_version(void);

/* Human-readable name of a status code. Never NULL. */
LOCKS_API const char* locks_status_string(int status);

/*
 * k_cap: row stride of `selected` = min(budget_tokens / 16, max_pages_per_seq),
 * at least 1. The number of pages kept per (sequence, kv head) is
 * k = min(budget_tokens / 16, seq_pages[b])  ([post] "Code": budget // page).
 * Returns LOCKS_ERR_INVALID_ARG for a null dims or a negative budget.
 */
LOCKS_API int locks_k_cap(const locks_dims_t* dims, int32_t budget_tokens, int32_t* k_cap);

/*
 * Workspace bytes needed by every call below for these dims and budget
 * (the decode step needs the most: the score table, its LSE partials, the
 * selection and the device status word; the split partials of
 * locks_sparse_attention share that space). The workspace must be 256-byte
 * aligned. Its first 256 bytes hold the status word; locks_clear_device_status
 * zeroes it. Its other contents are scratch between calls.
 */
LOCKS_API int locks_workspace_size(const locks_dims_t* dims, int32_t budget_tokens, size_t* bytes);

/*
 * Bytes of the lse_partials buffer of locks_score_pages / locks_select_pages /
 * locks_select_attend for these dims (16-byte aligned): one (max, sum exp) pair per
 * (sequence, query head, scoring CTA, consumer warp), the scoring grid being at most 256
 * CTAs. The selection reduces the per-head normaliser from them without reading the score
 * table or exchanging partial sums between its CTAs.
 */
LOCKS_API int locks_lse_partials_size(const locks_dims_t* dims, size_t* bytes);

/*
 * Summary build ([post] "How LOCKS works": a one-time decomposition of the
 * centred keys when a page fills, off the decode critical path; [summary] 2.1:
 * a small eigendecomposition of the centred keys, int8 centroid, int4 basis,
 * int8 coefficients, about 10% of the page's K/V bytes).
 * For each listed physical page p = phys_page_ids[i] (0 <= i < n_pages) and
 * each kv head: mu = mean of the 16 keys; D = K - mu; eigenpairs of the 16x16
 * Gram D D^T (descending); for the top 8: V[:, r] = D^T u_r / sqrt(lambda_r),
 * C[:, r] = sqrt(lambda_r) u_r, a column with lambda_r <= 1e-12 lambda_1 is
 * zero; the largest-magnitude entry of each V column is made positive; then
 * absmax-quantised into the summary layout above. Pages not listed are left
 * untouched. Computed in fp32 on the GPU.
 */
LOCKS_API int locks_build_summaries(const locks_dims_t* dims, const uint16_t* k_cache,
                                    const int32_t* phys_page_ids, int32_t n_pages,
                                    locks_summaries_t summaries, void* workspace,
                                    size_t workspace_bytes, void* stream);

/*
 * Page scores from the summaries alone ([post] "How LOCKS works" and
 * [summary] 2.2; no key or value is read):
 *   scores[b][h][j] = log sum_{i < 16} exp[(q.mu_j + (V_j^T q).c_i) / sqrt(128)]
 * for every sequence b, query head h and logical page j < seq_pages[b], with
 * the summary of unit (page_table[b][j], h / g) dequantised. Entries
 * j >= seq_pages[b] are not written. When lse_partials is not NULL it also
 * receives the (max, sum exp) of the scores per query head split by the scoring
 * CTA and warp (locks_lse_partials_size bytes), from which the selection forms the
 * per-head normaliser without re-reading the whole score table.
 */
LOCKS_API int locks_score_pages(const locks_dims_t* dims, const float* q, locks_summaries_t summaries,
                                const int32_t* page_table, const int32_t* seq_pages, float* scores,
                                float* lse_partials, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Group-shared top-k selection ([summary] 2.3: mean of the estimated mass
 * shares over the query heads of a GQA group; [post] "Code": keep
 * budget // 16 pages, indices sorted ascending).
 *   L_h   = log sum_{j < seq_pages[b]} exp(scores[b][h][j])
 *   key_j = log( (1/g) sum_{h in group} exp(scores[b][h][j] - L_h) )
 * selected[b][kvh][0..k) = the k logical pages with the largest key (radix
 * select on the order-preserving 32-bit image of key), equal keys ranked by
 * lower page id, NaN keys ranked below -inf, written in ascending order;
 * n_selected[b][kvh] = k. sel_keys (fp32 [B][Hkv][max_pages_per_seq], may be
 * NULL) receives key_j for j < seq_pages[b]. lse_partials (may be NULL) are
 * the partials locks_score_pages wrote for these same scores and dims on this
 * device; when given, L_h is reduced from them. A NaN score adds nothing to L_h and
 * gives its page a NaN key, which ranks last.
 */
LOCKS_API int locks_select_pages(const locks_dims_t* dims, const float* scores, const float* lse_partials,
                                 const int32_t* seq_pages, int32_t budget_tokens, int32_t* selected,
                                 int32_t* n_selected, float* sel_keys, void* workspace, size_t workspace_bytes,
                                 void* stream);

/*
 * Attention over the selected pages only ([post] "Code": scaled dot-product
 * attention of q over the keys/values of the chosen pages, scale 1/sqrt(128)):
 *   out[b][h] = sum_t softmax_t(q.k_t / sqrt(128)) v_t,  lse[b][h] = log sum_t exp(.)
 * over the 16 tokens of each page selected[b][h/g][0..n_selected[b][h/g]),
 * read through page_table. Split-K across the CTAs of a thread-block cluster
 * per (b, kv head), merged with the online-softmax rule. k_cap is the row
 * stride of `selected`. n = 0 gives out = 0 and lse = -inf.
 * With a workspace of at least locks_workspace_size(dims, 16 * k_cap) bytes
 * (any workspace of locks_workspace_size for these dims suffices in practice:
 * the split region is 256 + B*Hq*(4 + 4*130*4) bytes, rounded up), long
 * selections (>= 64 pages per CTA) are also split over up to 4 clusters per
 * (b, kv head) that stay co-resident; each writes its merged (m, l, o) to the
 * workspace and the last to arrive merges them (results equal the unsplit
 * launch up to the order of the merge). The call then zeroes the split
 * counters with an asynchronous memset on `stream` before the launch.
 */
LOCKS_API int locks_sparse_attention(const locks_dims_t* dims, const float* q, const uint16_t* k_cache,
                                     const uint16_t* v_cache, const int32_t* page_table,
                                     const int32_t* selected, const int32_t* n_selected, int32_t k_cap,
                                     uint16_t* out, float* lse, void* workspace, size_t workspace_bytes,
                                     void* stream);

/*
 * Selection and sparse attention fused in one cluster kernel: exactly
 * locks_select_pages followed by locks_sparse_attention on its result, in one
 * launch (the selection never leaves the cluster except through `selected`,
 * which the kernel writes and re-reads). selected is [B][Hkv][k_cap] with
 * k_cap = locks_k_cap(dims, budget_tokens); n_selected is [B][Hkv].
 */
LOCKS_API int locks_select_attend(const locks_dims_t* dims, const float* q, const uint16_t* k_cache,
                                  const uint16_t* v_cache, const int32_t* page_table, const float* scores,
                                  const float* lse_partials, const int32_t* seq_pages, int32_t budget_tokens,
                                  int32_t* selected, int32_t* n_selected, uint16_t* out, float* lse,
                                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * The whole decode step ([summary] 2.4: scoring, selection and sparse
 * attention captured together in CUDA graphs): locks_score_pages (with LSE
 * partials), then locks_select_attend.
 * scores, selected and n_selected may be NULL, in which case they live in the
 * workspace; when given they receive the same values as the separate calls.
 * Two kernel launches; no host synchronisation; graph-capturable.
 */
LOCKS_API int locks_decode_step(const locks_dims_t* dims, const float* q, const uint16_t* k_cache,
                                const uint16_t* v_cache, locks_summaries_t summaries,
                                const int32_t* page_table, const int32_t* seq_pages, int32_t budget_tokens,
                                uint16_t* out, float* lse, float* scores, int32_t* selected,
                                int32_t* n_selected, void* workspace, size_t workspace_bytes, void* stream);

/*
 * As locks_select_attend and locks_decode_step, plus each sequence's tokens that
 * have no summary yet. A page gets its summary only once it fills (LOCKS post,
 * "How LOCKS works": the decomposition runs when a page fills, every 16 tokens,
 * off the decode critical path), so the page being filled, and a filled page
 * whose summary is still being built, cannot be scored; their tokens are
 * attended whole, in the same softmax as the selected pages, and never selected.
 *   tail_tokens  int32 [batch], may be NULL (no tail): tail_tokens[b] in
 *                [0, 16 * LOCKS_MAX_TAIL_PAGES] tokens on logical pages
 *                seq_pages[b], seq_pages[b] + 1, ... (16 per page, the last one
 *                partial; physical pages through page_table, so the tail must end
 *                within max_pages_per_seq); other values record
 *                LOCKS_ERR_BAD_INDEX and the tail is skipped.
 * Page-fill refresh: when a page fills, the caller launches locks_build_summaries
 * for it (n_pages = 1) on another stream and keeps its 16 tokens in the tail
 * until that build has completed; then it advances seq_pages[b] by one and
 * takes 16 off tail_tokens[b]. With tail_tokens given, locks_decode_step_tail
 * runs its persistent scorer on one SM fewer than the GPU has, leaving that SM
 * to such a build (one CTA) instead of having a scorer CTA wait for it.
 */
LOCKS_API int locks_select_attend_tail(const locks_dims_t* dims, const float* q, const uint16_t* k_cache,
                                       const uint16_t* v_cache, const int32_t* page_table, const float* scores,
                                       const float* lse_partials, const int32_t* seq_pages,
                                       const int32_t* tail_tokens, int32_t budget_tokens, int32_t* selected,
                                       int32_t* n_selected, uint16_t* out, float* lse, void* workspace,
                                       size_t workspace_bytes, void* stream);
LOCKS_API int locks_decode_step_tail(const locks_dims_t* dims, const float* q, const uint16_t* k_cache,
                                     const uint16_t* v_cache, locks_summaries_t summaries,
                                     const int32_t* page_table, const int32_t* seq_pages,
                                     const int32_t* tail_tokens, int32_t budget_tokens, uint16_t* out, float* lse,
                                     float* scores, int32_t* selected, int32_t* n_selected, void* workspace,
                                     size_t workspace_bytes, void* stream);

/*
 * locks_decode_step without a workspace (the LOCKS pages have no counterpart
 * of this call; it exists for callers that cannot allocate device memory).
 * Serving engines usually reserve nearly all of HBM for their own paged KV
 * pool at start-up and give plugins no allocator, and cudaMalloc may
 * synchronise the device in the middle of a decode loop; such callers cannot
 * supply the workspace of locks_decode_step. Here the scratch (the score
 * table and the selection) lives in a fixed 36 MiB device array inside the
 * library, which every GPU that loads the library holds until the process
 * exits. The caller still passes all inputs and outputs (out, and lse which
 * may be NULL).
 * - Returns LOCKS_ERR_WORKSPACE_TOO_SMALL when locks_workspace_size(dims,
 *   budget_tokens) exceeds 36 MiB. The score table (4 bytes per sequence,
 *   query head and page) dominates: at 32 query heads and 65536 pages (1M
 *   tokens) each sequence needs 8 MiB of it plus 0.1-0.3 MiB of LSE partials,
 *   so batch 4 fits (32.5 MiB; 33 MiB with 2 kv heads) and batch 5 (40.6 MiB)
 *   is rejected.
 * - The first call in each CUDA context (per device) looks up the array's
 *   device address with that device current and caches it for that context;
 *   make that first call before any stream capture. Resetting the device
 *   (cudaDeviceReset) after that first call is not supported.
 * - All calls share the one array and it keeps the last call's contents:
 *   calls that overlap on the GPU (other streams, other threads) race and
 *   must be serialised by the caller.
 * - Device-side errors (bounded waits, bad page ids) are recorded in the
 *   array and cannot be read back by the caller; each call starts cleared.
 * - Calls no allocator (no cudaMalloc / cudaFree).
 */
LOCKS_API int locks_decode_step_noalloc(const locks_dims_t* dims, const float* q, const uint16_t* k_cache,
                                        const uint16_t* v_cache, locks_summaries_t summaries,
                                        const int32_t* page_table, const int32_t* seq_pages,
                                        int32_t budget_tokens, uint16_t* out, float* lse, void* stream);

/*
 * Copies the device status word (LOCKS_OK, LOCKS_ERR_TIMEOUT or
 * LOCKS_ERR_BAD_INDEX; the first error recorded wins) at the start of the
 * workspace to *status. Synchronises the stream.
 */
LOCKS_API int locks_get_device_status(const void* workspace, int32_t* status, void* stream);

/* Zeroes the device status word (asynchronous on stream). */
LOCKS_API int locks_clear_device_status(void* workspace, void* stream);

/*
 * Device-side bounded waits: sets the wall-time limit in nanoseconds that
 * every later launch from this process gives its mbarrier waits (0 restores
 * the default of 2 s). Host-side setting, read at launch time.
 */
LOCKS_API int locks_set_wait_limit_ns(uint64_t ns);

/*
 * Tuning and testing control (no counterpart on the LOCKS pages): pins the
 * thread-block cluster size of every later selection and attention launch from
 * this process (locks_select_pages, locks_sparse_attention, locks_select_attend,
 * locks_decode_step and their variants) to 8, 12 or 16 CTAs; 0 restores the
 * automatic choice. A 12-CTA cluster runs one CTA per SM; 8- and 16-CTA
 * clusters may run two. An attention-only launch that splits a long selection
 * over several clusters still picks its own size. Any other value returns
 * LOCKS_ERR_INVALID_ARG and changes nothing. A size whose shared memory does not
 * fit makes those launches return LOCKS_ERR_CUDA. The selection does not depend
 * on the size; the attention output does only through rounding (the share of
 * pages each warp accumulates). Host-side setting, read at launch time.
 */
LOCKS_API int locks_set_select_cluster(int32_t cluster);

/*
 * Failure-detection self test (no counterpart on the LOCKS pages): launches
 * one CTA that waits on an mbarrier phase nothing will complete. The wait
 * gives up after limit_ns and records LOCKS_ERR_TIMEOUT in the status word of
 * `workspace` (>= 256 bytes); the context stays usable. Asynchronous.
 */
LOCKS_API int locks_selftest_bounded_wait(void* workspace, size_t workspace_bytes, uint64_t limit_ns,
                                          void* stream);

/* ------------------------------------------------------------------------
 * Selector ablations (synthetic-carrier studies; not on the decode path).
 *
 * These calls score pages by other selectors than the shipped summary, for
 * recall and mass-coverage studies; the scores go through locks_select_pages
 * like the summary scores do. All take the decode step's dims, queries
 * (fp32 [B][Hq][128]), K cache (bf16 bits [num_phys_pages][Hkv][16][128],
 * 16-byte aligned), page table and seq_pages, and write fp32 scores
 * [B][Hq][max_pages_per_seq] for j < seq_pages[b] only (other entries are not
 * written). An out-of-range page-table entry is read as physical page 0 and
 * recorded as LOCKS_ERR_BAD_INDEX in the workspace status word when a
 * workspace is given. Asynchronous on `stream`; the caller owns every buffer.
 * ------------------------------------------------------------------------ */

/*
 * Bytes of workspace locks_shared_basis and locks_shared_scores need
 * (256-byte aligned): the status word, the fp32 second moments
 * [B][Hkv][128][128] and the projected queries [B][Hq][128].
 */
LOCKS_API int locks_ablation_workspace_size(const locks_dims_t* dims, size_t* bytes);

/*
 * Exact page scores, the selector that reads every key ([summary] sections
 * 1 and 3: exact selection reads all keys, the reference LOCKS is measured
 * against):
 *   scores[b][h][j] = log sum_i exp(q_h . k_i / sqrt(128)) over the 16 keys of
 *   physical page page_table[b][j], kv head h / (Hq / Hkv).
 * workspace may be NULL (then no status is recorded). Reads 4 KB per unit.
 */
LOCKS_API int locks_exact_scores(const locks_dims_t* dims, const float* q, const uint16_t* k_cache,
                                 const int32_t* page_table, const int32_t* seq_pages, float* scores,
                                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * Scores of page-local summaries of another rank or code width, built from the
 * keys and scored in one pass ([post] "Caveats": int4 loses a few recall
 * points, int2 collapses; [post] "How LOCKS works" for the summary and its
 * score; Theorem 1 covers the unquantised rank-r summary). Per unit: mu, the
 * top-`rank` eigenpairs of the centred keys' 16 x 16 Gram matrix (cyclic
 * Jacobi), V[:, r] = D^T u_r / sqrt(lambda_r), C[:, r] = sqrt(lambda_r) u_r
 * (zero where lambda_r <= 1e-12 lambda_1); mu, V and C are each replaced by
 * their symmetric absmax codes of bits_mu / bits_v / bits_c bits (scale =
 * fp16(absmax / (2^(bits-1) - 1)), round half to even), or kept when the
 * width is 0; then the summary score of locks_score_pages. rank 8 with widths
 * (8, 4, 8) is the shipped summary. rank must be 1..15 (15 spans the 16
 * centred keys), each width 0 or 2..8, else LOCKS_ERR_INVALID_ARG.
 */
LOCKS_API int locks_variant_scores(const locks_dims_t* dims, const float* q, const uint16_t* k_cache,
                                   const int32_t* page_table, const int32_t* seq_pages, int32_t rank,
                                   int32_t bits_mu, int32_t bits_v, int32_t bits_c, float* scores,
                                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * The shared basis a shared-projection selector builds from the full sequence
 * ([post] "Why shared-basis sparse attention is structurally broken"): per
 * (b, kv head), the `rank` (0..128) eigenvectors of largest eigenvalue of the
 * uncentred second moment M = sum_t k_t k_t^T over every token of the
 * sequence's seq_pages[b] pages (fp32, parallel cyclic Jacobi), written as
 * rows basis[b][kvh][r][128] (rank-major), each with its largest-magnitude
 * entry positive, zero where lambda_r <= 1e-12 lambda_1. eigvals (nullable)
 * receives all 128 eigenvalues of each M in descending order
 * ([B][Hkv][128]). workspace must hold locks_ablation_workspace_size bytes.
 */
LOCKS_API int locks_shared_basis(const locks_dims_t* dims, const uint16_t* k_cache, const int32_t* page_table,
                                 const int32_t* seq_pages, int32_t rank, float* basis, float* eigvals,
                                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * Shared-basis page scores ([post] "Why shared-basis sparse attention is
 * structurally broken"; Proposition 1, [summary] section 3): the
 * keys seen through the fixed projection P = W W^T of the basis W
 * (basis[b][kvh][rank][128], orthonormal rows, e.g. from locks_shared_basis),
 *   scores[b][h][j] = log sum_i exp(q_h . (P k_i) / sqrt(128)),
 * computed as the exact score of the projected query P q_h (P is symmetric).
 * A page whose keys lie in the null space of W^T scores log 16 for any query.
 * workspace must hold locks_ablation_workspace_size bytes.
 */
LOCKS_API int locks_shared_scores(const locks_dims_t* dims, const float* q, const uint16_t* k_cache,
                                  const int32_t* page_table, const int32_t* seq_pages, const float* basis,
                                  int32_t rank, float* scores, void* workspace, size_t workspace_bytes,
                                  void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LOCKS_H */
