/*
 * kvr.h -- C ABI of libkvr: decode-step KV page retrieval and sparse GQA
 * decode attention on one NVIDIA B300 (sm_103a).
 *
 * Sources of the operations (titles of the pages, section names):
 *   [FreeKV]  "FreeKV: Boosting KV Cache Retrieval for Efficient LLM
 *             Inference", technical summary: section 1 (Problem: KV retrieval
 *             keeps the whole cache and uses only the part each step needs),
 *             section 2.1 (Algorithm side: speculative retrieval, fine-grained
 *             correction, group-consistent similarity) and section 2.2
 *             (System side: hybrid NHD/HND layouts, streamed recall with
 *             double buffering).
 *   [KVwiki]  "Key-Value (KV) Cache" wiki page: decoding appends one token's
 *             K/V per step and is memory-bandwidth bound; PagedAttention
 *             stores the cache in fixed-size pages; grouped-query attention.
 * The pages describe selection by page but print no page-score formula.  This
 * library scores a page with the per-channel upper bound of q.k built from the
 * page's per-channel key minimum and maximum (kvr_build_summaries,
 * kvr_select_pages).
 *
 * Conventions for every call:
 *   - bf16 tensors are passed as `uint16_t*` holding raw bfloat16 bits;
 *     int32 and fp32 tensors as their own types.  All tensors are dense,
 *     row-major, in DEVICE memory unless stated otherwise, and must start on
 *     a 16-byte boundary.
 *   - Shapes: B = batch, Hq = query heads, H = KV heads, G = Hq / H query
 *     heads per KV head (query head h uses KV head h / G), D = head_dim,
 *     P = page_size, N = logical pages per sequence, k = top_k.
 *   - The K and V pools hold physical pages in token-major (NHD) order:
 *     [n_phys_pages][P][H][D]; page_table [B][N] maps a sequence's logical
 *     page to a physical page.
 *   - Supported: D = 128; G in {1, 2, 4, 8}; P in {16, 32, 64};
 *     1 <= k <= N <= 16384; H <= 64; B <= 65535.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every call only enqueues work on its stream(s) and returns;
 *     it never synchronises, except kvr_get_status and kvr_stream_wait.
 *   - The caller allocates and owns every buffer, workspace, state and
 *     stream.  The library allocates no device memory; its only device state
 *     is a 32-bit status word (see kvr_get_status).
 *   - Errors: a call returns KVR_OK (0) or a negative KVR_ERR_* code.
 *     Argument checks happen before any launch, so a rejected call enqueues
 *     nothing.  Conditions found on the device (an out-of-range page id, a
 *     wait that timed out) set bits of the status word instead.
 *   - A workspace (`ws`, `ws_bytes`) must be at least kvr_workspace_size()
 *     bytes.  Its contents need no initialisation: a call writes every
 *     scratch value before reading it, except the speculative step's one
 *     8-byte early-start word per (b, g) (kvr_speculative_step and
 *     kvr_speculative_step_host; other calls leave it as found).  The step's
 *     top-k sets a reused head's word to a 64-bit tag of the call (a fixed
 *     32-bit pattern above a per-process call count), the attention reads it
 *     and clears it: any other prior value is ignored, so only a stale word
 *     that happened to hold that exact tag could mislead a call.  Calls that
 *     share a workspace must not overlap on the GPU.
 */
#ifndef KVR_H
#define KVR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVR_OK 0
#define KVR_ERR_INVALID_ARG (-1)       /* null pointer, negative size, bad enum */
#define KVR_ERR_UNSUPPORTED_SHAPE (-2) /* a dimension outside the supported set */
#define KVR_ERR_ALIGN (-3)             /* a pointer not on a 16-byte boundary */
#define KVR_ERR_WORKSPACE (-4)         /* workspace missing or too small */
#define KVR_ERR_CUDA (-5)              /* a CUDA call or launch failed */
#define KVR_ERR_TIMEOUT (-6)           /* a host-side wait ran past its deadline */
#define KVR_ERR_SCRATCH_LIMIT (-7)     /* needs more than KVR_NOALLOC_SCRATCH_BYTES */

/* status-word bits set by kernels */
#define KVR_ST_BAD_INDEX 0x1u     /* a page id outside its pool was skipped */
#define KVR_ST_WAIT_TIMEOUT 0x2u  /* a kernel gave up waiting for a copy */
#define KVR_ST_NO_TOKENS 0x4u     /* an attention row had no valid token */
#define KVR_ST_NO_FREE_SLOT 0x8u  /* recall found fewer free slots than misses */

/* output element types of kvr_sparse_decode_attn_multi */
#define KVR_DTYPE_F32 0  /* fp32 */
#define KVR_DTYPE_BF16 1 /* bf16, the fp32 result rounded to nearest even once */

/* workspace kinds for kvr_workspace_size */
#define KVR_OP_SELECT 1 /* kvr_select_pages, kvr_speculative_select */
#define KVR_OP_ATTN 2   /* kvr_sparse_decode_attn */
#define KVR_OP_STEP 3   /* kvr_speculative_step(_overlap), kvr_speculative_step_recall */
#define KVR_OP_STEP_HOST 4 /* kvr_speculative_step_host */

typedef struct kvr_dims {
  int32_t batch;        /* B */
  int32_t n_q_heads;    /* Hq */
  int32_t n_kv_heads;   /* H */
  int32_t head_dim;     /* D */
  int32_t page_size;    /* P */
  int32_t n_pages;      /* N, logical pages per sequence */
  int32_t n_phys_pages; /* pages in the K/V pools */
} kvr_dims;

/* Bytes of workspace a call of kind `op` needs for these dims and top_k
 * (0 for invalid arguments). */
size_t kvr_workspace_size(const kvr_dims *dims, int32_t top_k, int32_t op);

/* Page summaries.  For every sequence b, KV head g and logical page p, the
 * per-channel minimum and maximum of the P keys of that page:
 *   summ[b][g][p][0][c] = min_t K[page_table[b][p]][t][g][c]
 *   summ[b][g][p][1][c] = max_t K[page_table[b][p]][t][g][c]
 * k_pool [n_phys][P][H][D] bf16; page_table [B][N] int32; summ
 * [B][H][N][2][D] bf16 (written; min and max of bf16 values are bf16, so the
 * summary is exact).  Pages are the paged cache of [KVwiki] (PagedAttention);
 * the summary feeds the page score of kvr_select_pages.  A page_table entry
 * outside [0, n_phys) sets KVR_ST_BAD_INDEX and leaves that summary
 * unwritten. */
int kvr_build_summaries(const kvr_dims *dims, const uint16_t *k_pool,
                        const int32_t *page_table, uint16_t *summ, void *stream);

/* KV selection for one decode step ([FreeKV] section 1: select the needed
 * part of the kept cache; section 2.1: selection per KV head, group-
 * consistent).  For each (b, g) the page score is
 *   S[b][g][p] = (1/G) * sum_{h in group g} sum_c max(q[b][h][c]*kmin_c, q[b][h][c]*kmax_c)
 * accumulated in fp32 from exact bf16 products, and the top_k pages with the
 * largest S are selected, ties to the lower page id.
 * q [B][Hq][D] bf16; summ from kvr_build_summaries; page_table [B][N].
 * Outputs: sel [B][H][k] int32 logical page ids in ascending order;
 * sel_phys [B][H][k] int32 = page_table[b][sel] (may be NULL); scores_opt
 * [B][H][N] fp32 copy of S (may be NULL).  Workspace kind KVR_OP_SELECT. */
int kvr_select_pages(const kvr_dims *dims, const uint16_t *q,
                     const uint16_t *summ, const int32_t *page_table,
                     int32_t top_k, int32_t *sel, int32_t *sel_phys,
                     float *scores_opt, void *ws, size_t ws_bytes, void *stream);

/* Sparse GQA decode attention over the selected pages ([FreeKV] section
 * 2.1: step i attends over the retrieved pages; [KVwiki]: GQA).  For query
 * head h of sequence b with KV head g = h / G, over the tokens t of pages
 * sel_phys[b][g][0..k) (physical ids into the pools):
 *   out[b][h] = sum_t softmax_t(scale * q[b][h] . K_t) * V_t
 * computed in fp32 (split over the selected pages, then merged with a
 * log-sum-exp rescale).  scale <= 0 means 1/sqrt(D).  q [B][Hq][D] bf16;
 * k_pool, v_pool [n_phys][P][H][D] bf16; sel_phys [B][H][k] int32; out
 * [B][Hq][D] fp32.  An id outside [0, n_phys) is skipped and sets
 * KVR_ST_BAD_INDEX.  Workspace kind KVR_OP_ATTN. */
int kvr_sparse_decode_attn(const kvr_dims *dims, const uint16_t *q,
                           const uint16_t *k_pool, const uint16_t *v_pool,
                           const int32_t *sel_phys, int32_t top_k, float scale,
                           float *out, void *ws, size_t ws_bytes, void *stream);

/* ---- partial last pages and decode-time append ([KVwiki]: each decode step
 * appends the new token's K and V; PagedAttention fills a sequence's pages
 * in order).  seq_len [B] int32 (device) counts the tokens sequence b has
 * written: it has started ceil(seq_len[b] / P) pages and logical page p
 * holds min(P, seq_len[b] - p P) tokens (rows 0 .. of the page). */

/* Append one token per sequence: for every KV head g, K row k_new[b][g] and
 * V row v_new[b][g] ([B][H][D] bf16) go to row t mod P of logical page t / P
 * (physical page page_table[b][t / P]) with t = seq_len[b]; that page's
 * summary in summ becomes the min/max over its written tokens (the new key
 * alone when it starts the page); then seq_len[b] = t + 1.  A sequence that
 * is full (t >= N P) or whose page id is outside [0, n_phys) is left as is
 * and sets KVR_ST_BAD_INDEX.  The caller maps the page before its first
 * token.  One kernel on `stream`. */
int kvr_append_kv(const kvr_dims *dims, const uint16_t *k_new,
                  const uint16_t *v_new, const int32_t *page_table,
                  int32_t *seq_len, uint16_t *k_pool, uint16_t *v_pool,
                  uint16_t *summ, void *stream);

/* kvr_build_summaries over the written tokens of each page only; pages a
 * sequence has not started are left untouched. */
int kvr_build_summaries_len(const kvr_dims *dims, const uint16_t *k_pool,
                            const int32_t *page_table, const int32_t *seq_len,
                            uint16_t *summ, void *stream);

/* kvr_select_pages over the started pages of each sequence only.  A
 * sequence with fewer started pages than top_k selects all of them
 * (ascending) and fills the rest of its rows of sel and sel_phys with -1.
 * Workspace kind KVR_OP_SELECT. */
int kvr_select_pages_len(const kvr_dims *dims, const uint16_t *q,
                         const uint16_t *summ, const int32_t *page_table,
                         const int32_t *seq_len, int32_t top_k, int32_t *sel,
                         int32_t *sel_phys, float *scores_opt, void *ws,
                         size_t ws_bytes, void *stream);

/* kvr_sparse_decode_attn over written tokens only: in the physical page
 * page_table[b][(seq_len[b] - 1) / P] (the sequence's last, possibly partial
 * page) only its written rows take part; a -1 entry of sel_phys is no page
 * (skipped without a status bit).  sel_phys must hold started pages.
 * Workspace kind KVR_OP_ATTN. */
int kvr_sparse_decode_attn_len(const kvr_dims *dims, const uint16_t *q,
                               const uint16_t *k_pool, const uint16_t *v_pool,
                               const int32_t *page_table, const int32_t *seq_len,
                               const int32_t *sel_phys, int32_t top_k,
                               float scale, float *out, void *ws,
                               size_t ws_bytes, void *stream);

/* ---- several query tokens per sequence in one step.  The pages treat one
 * new token per decode step; a step that decodes several (the T newest
 * tokens of each sequence, whose K and V are already appended) is this
 * library's extension of [FreeKV] section 2.1's group-consistent selection:
 * one selection per (b, g) serves the whole step, scored with the mean of
 * the page bound over every query row that will read the pages (the G heads
 * of the group times the T tokens), and each query token attends causally.
 * qs [B][T][Hq][D] bf16: the queries of the last T tokens of each sequence,
 * oldest first.  G T must be 1, 2, 4, 8 or 16 (KVR_ERR_UNSUPPORTED_SHAPE
 * otherwise).  seq_len [B] counts the written tokens including the T new
 * ones (seq_len[b] >= T). */

/* The step's selection: for each (b, g) the page score is
 *   S[b][g][p] = (1 / (T G)) * sum_{tau < T} sum_{h in group g} sum_c
 *                max(qs[b][tau][h][c]*kmin_c, qs[b][tau][h][c]*kmax_c)
 * over the sequence's started pages, and the top_k pages with the largest S
 * are selected as in kvr_select_pages_len (ties to the lower page id, ids
 * ascending, -1 beyond the started pages).  Workspace kind KVR_OP_SELECT. */
int kvr_select_pages_multi(const kvr_dims *dims, const uint16_t *qs,
                           int32_t n_query, const uint16_t *summ,
                           const int32_t *page_table, const int32_t *seq_len,
                           int32_t top_k, int32_t *sel, int32_t *sel_phys,
                           float *scores_opt, void *ws, size_t ws_bytes,
                           void *stream);

/* The step's attention: query token tau of sequence b (0 <= tau < T), head
 * h, attends over the tokens of its KV head's selected pages at positions
 * below seq_len[b] - T + tau + 1 (its own token and the ones before it):
 *   out[b][tau][h] = sum_t softmax_t(scale * qs[b][tau][h] . K_t) * V_t .
 * sel [B][H][k] holds the logical ids (from kvr_select_pages_multi; needed
 * for T > 1, may be NULL for T = 1) and sel_phys the physical ones.  out
 * [B][T][Hq][D] is fp32 (out_dtype KVR_DTYPE_F32) or bf16 (KVR_DTYPE_BF16:
 * the fp32 result rounded to nearest even once, at the store).  With T = 1
 * this is kvr_sparse_decode_attn_len with a choice of output type.  A row
 * that sees no token gets zeros and sets KVR_ST_NO_TOKENS.  Workspace kind
 * KVR_OP_ATTN. */
int kvr_sparse_decode_attn_multi(const kvr_dims *dims, const uint16_t *qs,
                                 int32_t n_query, const uint16_t *k_pool,
                                 const uint16_t *v_pool,
                                 const int32_t *page_table,
                                 const int32_t *seq_len, const int32_t *sel,
                                 const int32_t *sel_phys, int32_t top_k,
                                 float scale, void *out, int32_t out_dtype,
                                 void *ws, size_t ws_bytes, void *stream);

/* State of the speculative mode, owned by the caller.  q_prev [B][Hq][D]
 * bf16 and sel_prev [B][H][k] int32 are device buffers; `step` is a host
 * counter that the library increments on every successful step (0 before
 * the first).  Restoring the three restores the trace exactly. */
typedef struct kvr_spec_state {
  uint16_t *q_prev;
  int32_t *sel_prev;
  int32_t step;
} kvr_spec_state;

/* Speculative selection ([FreeKV] section 2.1).  Computes the selection of
 * the current query (as kvr_select_pages) and, per (b, g), the group
 * similarity C = mean over the group's query heads of cos(q_t, q_prev)
 * (fp32; cosine 0 for a zero vector).  The KV head is corrected when
 * step == 0 or C < tau; the selection used by this step is the current
 * query's for corrected heads and the previous step's (sel_prev) for the
 * others.  Then sel_prev <- current selection and q_prev <- q_t.
 * Outputs: corrected [B][H] uint8; cbar_opt [B][H] fp32 (may be NULL);
 * sel_used [B][H][k] logical ids ascending; sel_used_phys [B][H][k] =
 * page_table[b][sel_used] (may be NULL).  Workspace kind KVR_OP_SELECT.
 * Increments st->step on success. */
int kvr_speculative_select(const kvr_dims *dims, kvr_spec_state *st,
                           const uint16_t *q_t, const uint16_t *summ,
                           const int32_t *page_table, int32_t top_k, float tau,
                           uint8_t *corrected, float *cbar_opt,
                           int32_t *sel_used, int32_t *sel_used_phys,
                           void *ws, size_t ws_bytes, void *stream);

/* One speculative decode step: kvr_speculative_select followed by
 * kvr_sparse_decode_attn over sel_used_phys (which must be non-NULL), both on
 * `stream`.  The attention of a head that reuses its previous selection
 * starts as soon as the selection kernel has announced that head's page ids
 * (taken before the new selection is computed), without waiting for the
 * rest of the selection ([FreeKV] section 2.1: speculative retrieval takes
 * the selection off the critical path); results are unchanged.  Workspace
 * kind KVR_OP_STEP. */
int kvr_speculative_step(const kvr_dims *dims, kvr_spec_state *st,
                         const uint16_t *q_t, const uint16_t *summ,
                         const int32_t *page_table, const uint16_t *k_pool,
                         const uint16_t *v_pool, int32_t top_k, float tau,
                         float scale, float *out, uint8_t *corrected,
                         float *cbar_opt, int32_t *sel_used,
                         int32_t *sel_used_phys, void *ws, size_t ws_bytes,
                         void *stream);

/* kvr_speculative_step with the query and the output in host memory
 * ([FreeKV] section 2.2: the step's data movement stays off the critical
 * path).  q_host [B][Hq][D] bf16 and out_host [B][Hq][D] fp32 are
 * page-locked, mapped host memory (cudaHostAlloc, or cudaHostRegister with
 * mapping), 16-byte aligned; anything else returns KVR_ERR_INVALID_ARG
 * before any launch.  The call's first kernel copies q_host into the
 * workspace through the host mapping, and the attention stores the output
 * straight into out_host: no copy-engine transfer, so the step has no
 * hand-off between a copy and a kernel.  The first kernel may read q_host
 * before the kernel that precedes the call on `stream` has finished, so
 * q_host must hold the query when the call is made (written by the host, or
 * by device work already complete); the caller must not change q_host until
 * the call's work on `stream` has run, nor read out_host before then (an
 * event recorded after the call).  Results are bit-identical to
 * kvr_speculative_step on device copies of q and out.  Workspace kind
 * KVR_OP_STEP_HOST.  Increments st->step on success. */
int kvr_speculative_step_host(const kvr_dims *dims, kvr_spec_state *st,
                              const uint16_t *q_host, const uint16_t *summ,
                              const int32_t *page_table, const uint16_t *k_pool,
                              const uint16_t *v_pool, int32_t top_k, float tau,
                              float scale, float *out_host, uint8_t *corrected,
                              float *cbar_opt, int32_t *sel_used,
                              int32_t *sel_used_phys, void *ws, size_t ws_bytes,
                              void *stream);

/* The same speculative decode step with the selection taken off the
 * attention's critical path ([FreeKV] section 2.1: speculative retrieval
 * overlaps the selection with the computation).  On `stream`: the
 * correction decision per (b, g) (as in kvr_speculative_select), sel_used
 * and sel_used_phys of the reused heads from sel_prev, q_prev <- q_t; record
 * ev_decide.  On `side_stream`: wait ev_decide, score and select for the
 * current query (sel_prev <- the new selection; sel_used and sel_used_phys
 * of the corrected heads), record ev_select.  On `stream`: attention for
 * the reused heads (concurrently with the selection), wait ev_select,
 * attention for the corrected heads.  Results are bit-identical to
 * kvr_speculative_step.  ev_decide and ev_select are caller-created
 * cudaEvent_t passed as void*; sel_used_phys must be non-NULL.  Workspace
 * kind KVR_OP_STEP.  Increments st->step on success. */
int kvr_speculative_step_overlap(const kvr_dims *dims, kvr_spec_state *st,
                                 const uint16_t *q_t, const uint16_t *summ,
                                 const int32_t *page_table,
                                 const uint16_t *k_pool, const uint16_t *v_pool,
                                 int32_t top_k, float tau, float scale,
                                 float *out, uint8_t *corrected, float *cbar_opt,
                                 int32_t *sel_used, int32_t *sel_used_phys,
                                 void *ws, size_t ws_bytes, void *stream,
                                 void *side_stream, void *ev_decide,
                                 void *ev_select);

/* Host-resident cache for streamed recall ([FreeKV] section 2.2, hybrid
 * layouts: the host copy is head-major, HND).  k_host, v_host
 * [B][H][N][P][D] bf16 in page-locked host memory (cudaHostAlloc /
 * cudaHostRegister); each (b, g, p) page is one contiguous P*D block. */
typedef struct kvr_host_kv {
  const uint16_t *k_host;
  const uint16_t *v_host;
} kvr_host_kv;

/* Device working set of recalled pages.  k_slots, v_slots
 * [B][n_slots][P][H][D] bf16 (token-major, NHD, like the pools): slot s of
 * sequence b holds, for each KV head g separately, the page
 * slot2page[b][g][s].  page2slot [B][H][N] int32 (-1 = not resident) and
 * slot2page [B][H][n_slots] int32 (-1 = empty) are device maps.  n_slots
 * >= 2 * top_k (one set of slots read by the running step, one being
 * filled: double buffering). */
typedef struct kvr_working_set {
  uint16_t *k_slots;
  uint16_t *v_slots;
  int32_t *page2slot;
  int32_t *slot2page;
  int32_t n_slots;
} kvr_working_set;

/* Empty the working set's maps (all -1) on `stream`. */
int kvr_working_set_reset(const kvr_dims *dims, const kvr_working_set *wset,
                          void *stream);

/* Streamed recall ([FreeKV] section 2.2).  For every (b, g): the pages of
 * sel_new [B][H][k] that are not resident are copied from the host cache
 * into free slots, converting head-major host pages into the token-major
 * slot layout on the way (kernel loads read the page-locked host memory
 * directly).  Slots holding pages of sel_new or of protect [B][H][k] (the
 * selection the running attention reads) are never reused; free slots are
 * taken in ascending slot order for misses in ascending page order.  For
 * the heads with corrected[b][g] != 0 it also writes sel_slot_out[b][g][i] =
 * b * n_slots + page2slot[b][g][protect[b][g][i]] (for those heads protect
 * is the new selection itself).  n_copied_opt (device, may be NULL) is
 * incremented by the number of pages copied.  Runs on `stream` (normally a
 * side stream). */
int kvr_recall_pages(const kvr_dims *dims, const kvr_host_kv *host,
                     const kvr_working_set *wset, const int32_t *sel_new,
                     const int32_t *protect, const uint8_t *corrected,
                     int32_t top_k, int32_t *sel_slot_out,
                     uint32_t *n_copied_opt, void *stream);

/* One speculative decode step with the cache in host memory ([FreeKV]
 * sections 2.1 and 2.2).  On `stream`: speculative selection; the slots of
 * the non-corrected heads' reused pages (already resident) go to
 * sel_used_slot; record ev_select.  On `side_stream`: wait ev_select, recall
 * the current selection (protecting sel_used), record ev_recall.  On
 * `stream`: attention for the non-corrected heads (overlapping the recall),
 * wait ev_recall, attention for the corrected heads.  ev_select and ev_recall
 * are caller-created cudaEvent_t passed as void*.  The working set must have
 * been reset before the first step.  Workspace kind KVR_OP_STEP. */
int kvr_speculative_step_recall(const kvr_dims *dims, kvr_spec_state *st,
                                const uint16_t *q_t, const uint16_t *summ,
                                const kvr_host_kv *host,
                                const kvr_working_set *wset, int32_t top_k,
                                float tau, float scale, float *out,
                                uint8_t *corrected, float *cbar_opt,
                                int32_t *sel_used, int32_t *sel_used_slot,
                                uint32_t *n_copied_opt, void *ws,
                                size_t ws_bytes, void *stream,
                                void *side_stream, void *ev_select,
                                void *ev_recall);

/* ---- multi-layer decode pipeline ([FreeKV] section 2.1: the selection and
 * recall of a layer overlap that layer's attention and FFN and the next
 * layer's QKV projection; only heads that are corrected wait for them).
 *
 * One attention layer of a pipeline step.  The fields are those of the
 * single-layer calls: with host == NULL the layer's cache is HBM-resident
 * (page_table, k_pool, v_pool; sel_used_idx receives physical page ids, as
 * sel_used_phys of kvr_speculative_step_overlap); with host != NULL it is in
 * host memory (host, wset; sel_used_idx receives working-set slots, as
 * sel_used_slot of kvr_speculative_step_recall).  q is this step's query of
 * the layer.  ev are caller-created cudaEvent_t passed as void*, for a
 * host-resident layer (an HBM-resident one uses none; they may be NULL);
 * they carry the layer's dependencies from one pipeline step to the next,
 * so a layer keeps its events for the whole run (layers may share them).
 * Workspace kind KVR_OP_STEP; layers may share one workspace. */
typedef struct kvr_layer {
  kvr_spec_state *st;
  const uint16_t *q;
  const uint16_t *summ;
  const int32_t *page_table;
  const uint16_t *k_pool;
  const uint16_t *v_pool;
  const kvr_host_kv *host;
  const kvr_working_set *wset;
  float *out;
  uint8_t *corrected;
  float *cbar_opt;
  int32_t *sel_used;
  int32_t *sel_used_idx;
  uint32_t *n_copied_opt;
  void *ws;
  size_t ws_bytes;
  void *ev[3];
} kvr_layer;

/* Stand-in for the rest of each transformer layer.  A decode-time projection
 * is bound by reading its weights once, so each one is modelled by a kernel
 * that reads the same number of bytes: before a layer's selection, bytes
 * [0, qkv_bytes) of `weights` (the QKV projection); after its attention,
 * bytes [qkv_bytes, qkv_bytes + post_bytes) (the output projection and the
 * FFN).  Each read adds the 32-bit words it read, modulo 2^32, into *sink
 * (device).  qkv_bytes and post_bytes are multiples of 16, either may be 0,
 * and `weights` (device, 16-byte aligned) holds at least their sum. */
typedef struct kvr_stand_in {
  const void *weights;
  uint64_t qkv_bytes;
  uint64_t post_bytes;
  uint32_t *sink;
} kvr_stand_in;

/* One stand-in read on its own, on `stream`: bytes [offset, offset + bytes)
 * of compute->weights, summed into compute->sink (as the pipeline's reads;
 * for running the same model without the pipeline).  offset and bytes are
 * multiples of 16, and the range lies inside the caller's weights buffer. */
int kvr_stand_in_read(const kvr_stand_in *compute, uint64_t offset,
                      uint64_t bytes, void *stream);

/* Events a pipeline step records per layer when `marks` is given (index
 * layer * KVR_PIPE_MARKS + m), for a latency breakdown by
 * cudaEventElapsedTime:
 *   0 main, layer start           1 main, after the QKV stand-in
 *   2 main, after the speculative selection (host)
 *   3 main, after the reused heads' attention (host)
 *   4 main, once the side stream's work this layer waits for is done (host)
 *   5 main, after the corrected heads' attention (host) or the layer's
 *        attention (HBM)
 *   6 main, after the output/FFN stand-in
 *   7, 8 side stream: start and end of the recall of the corrected heads'
 *        pages (host)
 *   9, 10 prefetch stream: start and end of the recall of the other heads'
 *        pages for the next step (host)
 * An HBM layer runs its selection and attention as one chain of dependent
 * launches, which a mark between them would cut: it records 7 to 10 on the
 * main stream right after 1, and 2 to 4 right before 5 (its selection and
 * attention span 1 to 5). */
#define KVR_PIPE_MARKS 11

/* One decode step through n_layers attention layers, in layer order.  Per
 * layer, on `stream`: the QKV stand-in (if compute != NULL), then
 *   HBM-resident: kvr_speculative_step (the selection, whose speculative
 *     prologue lets the reused heads' attention start before it ends, then
 *     the attention), on `stream` alone;
 *   host-resident: a wait for this layer's prefetch of the previous step,
 *     the speculative selection, then on `side_stream` the recall of the
 *     corrected heads' pages and on `prefetch_stream` (after it) the recall
 *     of the other heads' new selection for the next step; the reused heads'
 *     attention beside them, a wait for the first recall only, the corrected
 *     heads' attention;
 * then the output/FFN stand-in.  Every layer's results are bit-identical to
 * kvr_speculative_step (HBM; also to kvr_speculative_step_overlap) or
 * kvr_speculative_step_recall (host) called layer by layer.  Every argument of every layer is checked before
 * anything is enqueued; a CUDA error part-way returns KVR_ERR_CUDA with the
 * work before it enqueued (st->step has advanced for every layer whose
 * selection was enqueued).  marks: NULL or
 * n_layers * KVR_PIPE_MARKS cudaEvent_t (created with timing); during a
 * stream capture they are recorded as external events, so the captured
 * graph records them on every replay (its last step leaves its times).  A host
 * layer's prefetch is joined to `stream` only by that layer's wait in the
 * next step: a caller that ends a CUDA-graph capture after a step, or needs
 * the working sets settled, first makes `stream` wait on each host layer's
 * ev[2].  That wait at the start of a step is on an event of the previous
 * step, and a capture may not wait on an event recorded outside it: a
 * caller that captures steps first records each host layer's ev[2] on the
 * capturing stream. */
int kvr_pipeline_step(const kvr_dims *dims, int32_t n_layers, kvr_layer *layers,
                      const kvr_stand_in *compute, int32_t top_k, float tau,
                      float scale, void *stream, void *side_stream,
                      void *prefetch_stream, void *const *marks);

/* Synchronise `stream`, then read and clear the device status word (a bit
 * set of KVR_ST_*).  Returns KVR_OK or KVR_ERR_CUDA.  A kernel still running
 * on another stream may set a bit between the read and the clear; for an
 * exact reading, let every stream that runs library kernels finish first. */
int kvr_get_status(void *stream, uint32_t *status_out);

/* Bound, in ns, of the kernels' waits for progress: a copy landing in
 * shared memory, a ring stage being released (0 restores the default, 2 s).
 * When such a wait runs out the kernel sets KVR_ST_WAIT_TIMEOUT, stops
 * issuing copies, waits for the copies it already issued (always with the
 * 2 s bound, so no copy is left in flight) and returns; the outputs of that
 * call are then unspecified and the context stays usable.  For tests of that
 * path, and for callers that want a hung copy engine reported sooner.  The
 * bound is a process-wide host setting passed to every launch enqueued
 * after the call (a captured graph keeps the bound of its capture).
 * Returns KVR_OK. */
int kvr_set_wait_limit(uint64_t ns);

/* Bounded host-side wait: return once all work enqueued on `stream` has
 * finished, or after timeout_us microseconds of host time, whichever comes
 * first (polling cudaStreamQuery; the thread yields between polls).
 * Returns KVR_OK when the stream is idle, KVR_ERR_TIMEOUT when the deadline
 * passed first (the work keeps running; the caller may wait again or give
 * up on it), KVR_ERR_CUDA when the stream reports an error.  timeout_us = 0
 * polls once. */
int kvr_stream_wait(void *stream, uint64_t timeout_us);

/* Static description of an error code (never NULL).  For KVR_ERR_CUDA the
 * text of the last CUDA error seen by the library is appended. */
const char *kvr_error_string(int code);

/* Bytes of a full K and V cache of one sequence:
 *   2 * n_layers * n_kv_heads * head_dim * n_tokens * bytes_per_elem.
 * ([KVwiki]: the cache grows linearly with context.)  0 on overflow or a
 * negative argument. */
uint64_t kvr_kv_bytes(int64_t n_layers, int64_t n_kv_heads, int64_t head_dim,
                      int64_t n_tokens, int64_t bytes_per_elem);

/* Allocation-free page selection.  The pages have no counterpart to this
 * entry point: it exists for callers that cannot allocate device memory,
 * such as an inference-engine plugin whose enqueue step may only use the
 * buffers it was handed, a serving loop that forbids allocation after
 * warm-up to keep latency flat, or a foreign-language caller with no access
 * to the process's device allocator.  It computes exactly what
 * kvr_select_pages computes (same kernels, same results), but its scratch
 * (the fp32 score rows) lives in a fixed array of
 * KVR_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that loads
 * the library keeps until the process exits.  The caller still passes all
 * inputs and outputs (q, summ, page_table, sel, sel_phys, scores_opt as in
 * kvr_select_pages).
 *   - Limit: the scratch is the score rows, B * H * N * 4 bytes, plus one
 *     4-byte word per (b, g), each part rounded up to a multiple of 256
 *     bytes: round256(B*H*N*4) + round256(B*H*4) <= KVR_NOALLOC_SCRATCH_BYTES
 *     (about one million page scores; B*H = 64 allows N up to 16383).
 *     Larger problems return KVR_ERR_SCRATCH_LIMIT before anything is
 *     enqueued.
 *   - Every call looks up the array's device address on the current device
 *     (a host-side query; it allocates nothing and stays valid across a
 *     cudaDeviceReset).  The first call on a device may make the driver load
 *     the library's device code, so make that first call before any stream
 *     capture.
 *   - All calls share the one array, which keeps the last call's contents
 *     (every score is written before it is read, so no call depends on
 *     them): calls that overlap on the GPU (on different streams, or from
 *     several threads) race and must be serialised by the caller.
 * It never calls cudaMalloc, cudaFree or any allocating routine. */
#define KVR_NOALLOC_SCRATCH_BYTES 4194304u /* 4 MiB */
int kvr_select_pages_noalloc(const kvr_dims *dims, const uint16_t *q,
                             const uint16_t *summ, const int32_t *page_table,
                             int32_t top_k, int32_t *sel, int32_t *sel_phys,
                             float *scores_opt, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KVR_H */
