/*
 * puzzlekv.h -- C ABI of the GB300 (sm_103a) PuzzleKV hot path.
 *
 * Page-wise low-rank KV cache compression as described in "PuzzleKV:
 * Page-Wise Low-Rank Decomposition for KV Cache Compression" (cited below as
 * [PuzzleKV] with its section and equation numbers):
 *   - every completed page of P tokens of each layer's per-KV-head key and
 *     value cache, outside a dense sink page and a dense local window, is
 *     factorized into rank-r factors L (P x r, orthonormal columns) and
 *     R = L^T X (r x d), through the P x P Gram matrix and its top-r
 *     eigenvectors                                  [PuzzleKV §3.3 ①②③, eq. (2)]
 *   - decode attention runs directly over dense and factorized pages with one
 *     online softmax, never reconstructing a page   [PuzzleKV §3.3 ④, eqs. (4)-(5)]
 *   - each decoded token is appended to the newest dense page; a page that
 *     leaves the local window is factorized once    [PuzzleKV §3.3 ⑤]
 *
 * Conventions shared by every entry point:
 *   - All functions are extern "C", never throw and never abort; they return a
 *     puzzlekv_status.  puzzlekv_last_error() gives a message for the calling
 *     thread's most recent failure.
 *   - Arguments are checked on the host before anything is launched; on a
 *     host-side error nothing is launched and no store state changes.
 *   - Device work is asynchronous on the given stream (a cudaStream_t passed
 *     as void*; NULL = legacy default stream).  A CUDA error raised by a
 *     launch is returned as PUZZLEKV_ERR_CUDA.
 *   - "device" pointers must point to memory of the current CUDA device and be
 *     16-byte aligned.  "host" pointers are read before the call returns.
 *   - The caller allocates and frees every device buffer; the library only
 *     borrows them.  It allocates no device memory itself.
 *   - Storage dtype: PUZZLEKV_BF16 (bf16 dense pages and factors, tensor-core
 *     path) or PUZZLEKV_F32 (fp32, CUDA-core path).  Outputs are fp32.
 *   - Supported shapes: head_dim d in {64, 128}; page size P in {16, 32, 64}
 *     with P <= d; 1 <= rank <= P; query heads per KV head G = Hq / H in
 *     1..8.  Key/value ranks are stored padded to a multiple of 8 (the
 *     padding is zero and never changes a result).
 *   - Calls that take a list of sequences (seq_ids, B) take 1 <= B <= 64
 *     distinct slots in [0, max_batch); an empty list is an invalid argument.
 */
#ifndef PUZZLEKV_H
#define PUZZLEKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PUZZLEKV_OK = 0,
    PUZZLEKV_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad index or size */
    PUZZLEKV_ERR_UNSUPPORTED = 2,   /* shape outside the supported set above */
    PUZZLEKV_ERR_CAPACITY = 3,      /* sequence would exceed max_tokens_per_seq */
    PUZZLEKV_ERR_NOT_CONVERGED = 4, /* an eigensolve hit its iteration cap (results kept) */
    PUZZLEKV_ERR_CUDA = 5,          /* a CUDA launch or copy failed */
    PUZZLEKV_ERR_DEVICE_TIMEOUT = 6 /* a kernel's bounded wait ran out (error flag set) */
} puzzlekv_status;

typedef enum { PUZZLEKV_F32 = 0, PUZZLEKV_BF16 = 1 } puzzlekv_dtype;

/* Page kinds as stored in the page table [PuzzleKV §3.3 ①②③]. */
enum { PUZZLEKV_PAGE_FACTORED = 0, PUZZLEKV_PAGE_DENSE = 1 };

/*
 * Store configuration.  sink_tokens: the first tokens kept dense; the sink
 * is every page holding one of them.  recent_tokens: width W of the dense
 * local window; every page holding one of the last W tokens stays dense, and
 * so does the incomplete last page [PuzzleKV §3.3 ①②③].  max_batch: number
 * of sequence slots.  max_tokens_per_seq: capacity per sequence.  A bf16
 * store's factor records must fit the decode kernel's shared-memory slots:
 * at page_size 64 and head_dim 128, rank_k + rank_v (each rounded up to a
 * multiple of 8) may be at most 72 (PUZZLEKV_ERR_UNSUPPORTED otherwise).
 * factor_int4: 0 = factors stored in kv_dtype; 1 = INT4 factors
 * [PuzzleKV §4.3]: singular values absorbed into both factors
 * (L = U Sigma^{1/2}, R = Sigma^{1/2} W^T), symmetric 4-bit codes in [-7, 7]
 * with one fp16 scale per column of L_K, R_K, R_V and per row of L_V.
 * Requires kv_dtype = PUZZLEKV_BF16 and rank_k, rank_v <= page_size / 2.
 * rope_theta: 0 = keys are stored as given (already rotated by the model's
 * RoPE, or without one) [PuzzleKV §4.1: post-RoPE keys].  > 0 = keys are
 * given before RoPE (prefill, append, decode step); pages are factorized
 * unrotated and every key is turned at attention by its absolute position n
 * with the rotate-half pairing (i, i + head_dim/2) and angles
 * n * rope_theta^(-2i/head_dim) [PuzzleKV Appendix D.3]; queries are given
 * already rotated at their own position.  Requires kv_dtype = PUZZLEKV_BF16,
 * factor_int4 = 0 and page_size 32 or 64.
 */
typedef struct {
    int32_t num_layers;
    int32_t num_kv_heads;
    int32_t num_q_heads;
    int32_t head_dim;
    int32_t page_size;
    int32_t rank_k;
    int32_t rank_v;
    int32_t sink_tokens;
    int32_t recent_tokens;
    int32_t max_batch;
    int32_t max_tokens_per_seq;
    int32_t kv_dtype; /* puzzlekv_dtype */
    int32_t factor_int4;
    float rope_theta;
} puzzlekv_config;

typedef struct puzzlekv_store puzzlekv_store; /* opaque host handle */

/*
 * Byte sizes of the four device buffers a store borrows for `cfg`:
 *   dense_pool: dense pages (sink, window, page being filled) for every
 *               (layer, sequence, KV head), K and V;
 *   factor_pool: one preallocated factor record per (layer, sequence, KV
 *               head, page) [PuzzleKV §3.3 ⑤: factors go to storage
 *               set aside in advance];
 *   page_table: per (sequence, layer): current length and one descriptor
 *               per page (kind, slot);
 *   workspace:  split-K partial softmax states and the device status word
 *               (for rope_theta > 0 also the fp32 (cos, sin) tables of the
 *               RoPE angles, filled by puzzlekv_store_create).
 * Host-only; needs no GPU.
 */
puzzlekv_status puzzlekv_query_sizes(const puzzlekv_config *cfg, size_t *dense_pool_bytes,
                                     size_t *factor_pool_bytes, size_t *page_table_bytes,
                                     size_t *workspace_bytes);

/*
 * Create a store over caller-allocated device buffers of at least the sizes
 * puzzlekv_query_sizes reports (all 256-byte aligned).  The buffers stay owned
 * by the caller and must outlive the store.  The call zero-fills the dense
 * pool, page table and workspace on `stream` (the factor pool is written
 * before it is read).  All sequence slots start empty.
 */
puzzlekv_status puzzlekv_store_create(const puzzlekv_config *cfg, void *dense_pool, void *factor_pool,
                                      void *page_table, void *workspace, void *stream,
                                      puzzlekv_store **out);

/* Free the host handle (not the device buffers). NULL is accepted. */
puzzlekv_status puzzlekv_store_destroy(puzzlekv_store *store);

/*
 * Prefill compression of one sequence [PuzzleKV §3.3 ①②③]: given its dense
 * prompt cache, partition every layer and KV head into pages, copy the dense
 * pages (sink, local window, incomplete last page) into the dense pool and
 * factorize every other page -- all layers, heads, keys and values in one
 * batched launch -- into the factor pool.
 *   k, v: device, [num_layers][num_kv_heads][T][head_dim] in kv_dtype,
 *         read-only, may be freed once the stream passes this call.
 *   seq:  sequence slot in [0, max_batch); any previous content is dropped.
 *   T:    prompt length, 1 <= T <= max_tokens_per_seq.
 */
puzzlekv_status puzzlekv_load_prefill(puzzlekv_store *store, int32_t seq, const void *k, const void *v,
                                     int32_t T, void *stream);

/*
 * Factorize a chosen list of completed pages [PuzzleKV §3.3 ③ and ⑤: every
 * completed page is factorized independently, once]: for each listed
 * (seq_ids[i], page_ids[i]), the key and value pages of every layer and KV
 * head, read from the dense pool, go into their preallocated factor records
 * in one batched launch on `stream`.  The page keeps its kind: a page inside
 * the local window stays dense for attention until it leaves the window,
 * which then only switches it to its factors (as puzzlekv_convert_ready_pages
 * does in the background).  Pages that already have factors are skipped
 * (never refactorized), and so is a page listed twice.
 *   seq_ids, page_ids: host, n entries.  A page must be complete (all P of
 *            its tokens present) in every layer of its sequence and must not
 *            be a sink page; any other entry (bad slot, empty sequence,
 *            incomplete, sink or out-of-range page) makes the call return
 *            PUZZLEKV_ERR_INVALID_ARG with nothing launched and no state
 *            changed.
 *   n:       number of entries; n = -1 ignores the lists (which may be NULL)
 *            and factorizes every eligible page (complete, not a sink page,
 *            no factors yet) of every sequence; n = 0 does nothing.
 * The call orders `stream` after any pending background conversion batch.
 */
puzzlekv_status puzzlekv_factorize_pages(puzzlekv_store *store, const int32_t *seq_ids, const int32_t *page_ids,
                                         int32_t n, void *stream);

/*
 * Prefill compression of one layer of one sequence, for prompt processing
 * that produces the cache layer by layer [PuzzleKV §3.3 ①②③, §4.5 time to
 * first token]: as puzzlekv_load_prefill restricted to `layer`.  The dense
 * pages and the page table are written on `stream`.  With async = 0 the
 * factorization also runs on `stream`.  With async = 1 it runs on the
 * store's internal low-priority stream, after the work already queued on
 * `stream`, so that the caller's next layers (their dense attention) overlap
 * it; the sequence's next attention call waits for it.
 *   k, v: device, [num_kv_heads][T][head_dim] in kv_dtype.  With async = 0
 *         they may be freed once the stream passes this call; with async = 1
 *         they are read on the internal stream (puzzlekv_background_stream),
 *         so they must stay unchanged until work queued there completes --
 *         order their reuse after puzzlekv_wait_background, or tell the
 *         allocator that owns them about that stream.
 *   seq, T: as puzzlekv_load_prefill; every layer of a sequence must be
 *         given the same T before it is decoded.
 */
puzzlekv_status puzzlekv_factorize_layer(puzzlekv_store *store, int32_t seq, int32_t layer, const void *k,
                                         const void *v, int32_t T, int32_t async, void *stream);

/* Make `stream` wait for all background work of the store (batched
 * conversions and asynchronous layer prefills) queued so far. */
puzzlekv_status puzzlekv_wait_background(puzzlekv_store *store, void *stream);

/* The store's internal low-priority stream (created on first use); owned by
 * the store and destroyed with it. */
puzzlekv_status puzzlekv_background_stream(puzzlekv_store *store, void **stream);

/*
 * Stateless batched page factorization [PuzzleKV §3.3 ③ and eq. (2)]:
 * for each of n independent pages X_i (P x d), G_i = X_i X_i^T in fp32, its
 * top-r eigenvectors, L_i (P x r, unit columns), and R_i = L_i^T X_i (r x d).
 * The eigensolve runs in fp32: a Householder reduction to tridiagonal form,
 * then, for r <= P / 2, multisection on Sturm counts for the eigenvalues
 * and inverse iteration with partial pivoting for the r vectors, or, for
 * r > P / 2, implicit QL with Wilkinson shifts on every eigenpair.
 *   X:      device, [n][P][d] in x_dtype (row = token).
 *   L, R:   device, [n][P][r] and [n][r][d] in out_dtype.
 *   sigma:  device fp32 [n][P] or NULL: sqrt of the eigenvalues (clamped at
 *           0), descending -- the singular values of X_i.
 *   status: device int32 or NULL; on return of the stream work, nonzero if
 *           an eigenvalue of any page took more than 30 QL iterations (r > P
 *           / 2 only; its factors are still written).
 */
puzzlekv_status puzzlekv_factorize_batch(const void *X, int32_t x_dtype, int64_t n, int32_t P, int32_t d,
                                         int32_t r, void *L, void *R, int32_t out_dtype, float *sigma,
                                         int32_t *status, void *stream);

/*
 * Byte size of one INT4 factor record of a store with these page size, head
 * dimension and ranks [PuzzleKV §4.3] (the `records` stride of
 * puzzlekv_factorize_batch_int4).  Host-only.
 */
puzzlekv_status puzzlekv_int4_record_bytes(int32_t P, int32_t d, int32_t rank_k, int32_t rank_v, int64_t *bytes);

/*
 * Stateless INT4 factorization of independent pages [PuzzleKV §4.3], the
 * computation an INT4 store runs on each page: the rank-r factorization of
 * puzzlekv_factorize_batch with every kept pair converged, singular values
 * absorbed into both factors (L~ = U Sigma^{1/2}, R~ = Sigma^{1/2} W^T), and
 * each factor quantized symmetrically to codes in [-7, 7] with fp16 scales
 * (max |x| / 7 per group; code = x / scale rounded to nearest even, clamped).
 *   X:       device bf16 [n][P][d].
 *   kind:    0 = key pages (rank rank_k; groups: columns of L~ and of R~),
 *            1 = value pages (rank rank_v; groups: rows of L~, columns of R~).
 *   records: device, [n][puzzlekv_int4_record_bytes(P, d, rank_k, rank_v)]:
 *            each page's code stream and scales for `kind` in the store's
 *            record layout; the other kind's bytes are not written.
 *   L_absorbed, R_absorbed: device fp32 [n][P][rp] and [n][rp][d] (rp = the
 *            rank rounded up to a multiple of 8, padding zero), or NULL: the
 *            absorbed factors the codes quantize, for checking the codes.
 *   status:  device int32 or NULL, nonzero if an eigensolve hit its cap.
 * Requires rank_k, rank_v <= P / 2 and the shapes of puzzlekv_factorize_batch.
 */
puzzlekv_status puzzlekv_factorize_batch_int4(const void *X, int64_t n, int32_t P, int32_t d, int32_t rank_k,
                                              int32_t rank_v, int32_t kind, void *records, float *L_absorbed,
                                              float *R_absorbed, int32_t *status, void *stream);

/*
 * Append one decoded token per listed sequence to `layer` [PuzzleKV §3.3 ⑤]:
 * the new key/value rows go into the newest dense page and take part in the
 * next attention call at once.  When the append moves a completed page out
 * of the local window, that page (keys and values of every KV head of this
 * layer) is factorized on `stream` into its preallocated factor record and
 * its dense slot is released -- at most one page per (sequence, layer) per
 * call; factorized pages are never revisited.
 *   k, v:    device, [B][num_kv_heads][head_dim] in kv_dtype.
 *   seq_ids: host, B distinct sequence slots, each already holding a prompt.
 */
puzzlekv_status puzzlekv_append_token(puzzlekv_store *store, int32_t layer, const void *k, const void *v,
                                      const int32_t *seq_ids, int32_t B, void *stream);

/*
 * Decode attention of one layer over the hybrid cache [PuzzleKV §3.3 ④]:
 * for each listed sequence and query head, softmax(q K^T / sqrt(d)) V over all
 * T cached tokens, with factorized pages evaluated as (q R_K^T) L_K^T and
 * (p L_V) R_V (eq. (4)) and all pages merged by one online softmax (eq. (5)).
 * Query head h reads KV head h / G.
 *   q:       device, [B][num_q_heads][head_dim] in kv_dtype.
 *   out:     device fp32, [B][num_q_heads][head_dim].
 *   seq_ids: host, B distinct sequence slots with T >= 1.
 */
puzzlekv_status puzzlekv_decode_attention(puzzlekv_store *store, int32_t layer, const void *q, float *out,
                                          const int32_t *seq_ids, int32_t B, void *stream);

/*
 * Factorize ahead of time, in batched launches over all sequences and
 * layers, the pages that are complete but have no factors yet (pages inside
 * the local window included) [PuzzleKV §3.3 ⑤].  A page's content is final
 * once its P tokens are present, W tokens before it leaves the window; when
 * it leaves, puzzlekv_append_token / puzzlekv_decode_step then only switch it
 * to its factors instead of factorizing one page per layer on the critical
 * path.  Calling this is optional (without it those calls factorize the page
 * themselves) and cheap when nothing is pending (host bookkeeping only);
 * calling it once per decode step, after the last layer, is the intended use.
 * Pages whose dense slot might be reused are never listed: a page reaches
 * the window's end before its slot comes round again.
 *   Pacing: a call starts a new batch only when the store's previous batch
 *   has finished, and a batch takes the pages nearest their leaving the
 *   window first, up to about one CTA per SM (num_SMs / (2 num_kv_heads)
 *   pages of all heads, keys and values).  Pages within 8 steps of leaving
 *   the window are always taken.  So a page may be converted a few calls
 *   after it completes, and the page jobs reach the SMs in small numbers
 *   beside the decode launches instead of all at once.
 *   Ordering: a batch runs on a low-priority stream internal to the store,
 *   after everything already queued on `stream`, one CTA per page job, so
 *   that it overlaps the decode steps that follow instead of stalling them.
 *   A batch's factors are first read when one of its pages becomes
 *   factorized; the first decode call (puzzlekv_decode_attention,
 *   puzzlekv_decode_step, the static-scratch variant) that reaches that
 *   length, and any prefill call (puzzlekv_load_prefill,
 *   puzzlekv_factorize_layer) that rewrites one of the batch's layers, makes
 *   its own stream wait for the batch.  puzzlekv_check_device_status and
 *   puzzlekv_factorize_counters synchronise the internal stream as well; the
 *   store must not be destroyed while its caller's streams still hold work
 *   that waits on a batch.
 */
puzzlekv_status puzzlekv_convert_ready_pages(puzzlekv_store *store, void *stream);

/*
 * One decode step of one layer in a single attention launch [PuzzleKV §3.3
 * ④ and ⑤]: append the new key/value row of each listed sequence (as
 * puzzlekv_append_token) and attend over the grown cache (as
 * puzzlekv_decode_attention), the new token included.  If the append moves a
 * completed page out of the local window, that page is factorized on
 * `stream` first, so this step already attends over its factors.
 *   q:   device, [B][num_q_heads][head_dim];  k, v: device, [B][num_kv_heads][head_dim]
 *   out: device fp32, [B][num_q_heads][head_dim]; seq_ids: host, B distinct slots.
 * Equivalent to puzzlekv_append_token followed by puzzlekv_decode_attention.
 */
puzzlekv_status puzzlekv_decode_step(puzzlekv_store *store, int32_t layer, const void *q, const void *k,
                                     const void *v, float *out, const int32_t *seq_ids, int32_t B, void *stream);

/*
 * Same computation and arguments as puzzlekv_decode_attention, for callers
 * that cannot allocate device memory where they decode (runtimes that forbid
 * allocation once serving has started, so that their footprint stays fixed
 * and no request fails on or waits for the allocator; embedders whose device
 * memory is owned by an allocator this layer cannot reach).  The page has no
 * counterpart: this is a deployment variant, not part of the method.
 *   - The split-K scratch (partial softmax states and split tickets) comes
 *     from a 16 MiB array compiled into the library, one per GPU that loads
 *     it, kept until the process exits; the store's workspace is not used
 *     for it.  Nothing is allocated by this call.
 *   - Stores needing more than 16 MiB of scratch (8 bytes x max_batch x
 *     num_kv_heads rounded up to 256 bytes, + 4 bytes x max_batch x
 *     num_q_heads x 128 x (head_dim + 4)) are rejected with
 *     PUZZLEKV_ERR_CAPACITY before anything is launched.  At head_dim 128
 *     that allows max_batch up to 7 with 32 query heads, 3 with 64 and 31
 *     with 8; at head_dim 64, 15 with 32 query heads.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current.  Under CUDA's lazy
 *     module loading (the default) that lookup is also what loads the
 *     library's device code on the device, and with it the 16 MiB array, so
 *     the first call can take device memory: make it once as a warm-up,
 *     before serving starts and before any stream capture begins.  Later
 *     calls take none.
 *   - Every call shares the one array and clears its counters on `stream`
 *     before launching; calls whose kernels overlap on the GPU
 *     (other streams, other threads) race on it and must be serialised by
 *     the caller.
 */
puzzlekv_status puzzlekv_decode_attention_static_scratch(puzzlekv_store *store, int32_t layer, const void *q,
                                                         float *out, const int32_t *seq_ids, int32_t B,
                                                         void *stream);

/*
 * Host-side accounting of one (sequence, layer) from the store's host mirror
 * (no device access): current length, dense and factorized page counts, and
 * the bytes those pages occupy (factors at the configured ranks plus the valid
 * rows of dense pages) [PuzzleKV §4.5 Memory Footprint].
 */
puzzlekv_status puzzlekv_store_stats(const puzzlekv_store *store, int32_t seq, int32_t layer, int32_t *length,
                                     int64_t *dense_pages, int64_t *factored_pages, int64_t *bytes_live);

/*
 * Test hook of the failure path (the page has no counterpart).  The store's
 * next decode launch (puzzlekv_decode_attention, puzzlekv_decode_step or the
 * static-scratch variant; bf16 stores) makes one of its shared-memory
 * barriers expect 16 bytes that no copy delivers, so that a bounded wait
 * runs out after wait_ns nanoseconds instead of the library's 1 s:
 *   where = 1: the first unit that the first CTA of the first listed
 *              sequence's KV head 0 streams; that CTA gives up, lets its
 *              copies land and exits without its split state, so no output
 *              row of that KV head is written;
 *   where = 2: the split merge of every (sequence, KV head) whose split
 *              states are staged in shared memory (all but calls with more
 *              splits than its room holds); those output rows are not
 *              written;
 *   where = 0: clears a pending request.
 * Nothing faults and nothing hangs: the launch ends (the drain of an
 * abandoned barrier is itself bounded by 1 s) and the next
 * puzzlekv_check_device_status returns PUZZLEKV_ERR_DEVICE_TIMEOUT and
 * clears the split tickets, after which the store decodes normally.  The
 * request applies to one launch.  wait_ns in [1e3, 1e9].
 */
puzzlekv_status puzzlekv_debug_fail_next_wait(puzzlekv_store *store, int32_t where, int64_t wait_ns);

/*
 * Synchronise `stream`, read the device status word and clear it.  Returns
 * PUZZLEKV_ERR_NOT_CONVERGED if an eigensolve hit its iteration cap since the last
 * check, PUZZLEKV_ERR_DEVICE_TIMEOUT if a kernel's bounded wait ran out.
 */
puzzlekv_status puzzlekv_check_device_status(puzzlekv_store *store, void *stream);

/*
 * Synchronise `stream`, then read and clear the store's factorization
 * counters: page jobs factorized (one K or one V page each) and the QL
 * plane rotations their eigensolves applied (jobs of rank above P / 2: a
 * smaller rank takes its top eigenpairs without QL), summed over every
 * factorization launch of the store (prefill, per-step and batched
 * conversion) since the last call.  For throughput accounting (the page has
 * no counterpart).  page_jobs and ql_rotations: host pointers, both
 * required.  The status flags read by
 * puzzlekv_check_device_status are left untouched.
 */
puzzlekv_status puzzlekv_factorize_counters(puzzlekv_store *store, void *stream, int64_t *page_jobs,
                                            int64_t *ql_rotations);

/*
 * Host-only page classification, the rule the store and its kernels apply
 * [PuzzleKV §3.3 ①②③, ⑤]: writes PUZZLEKV_PAGE_DENSE or
 * PUZZLEKV_PAGE_FACTORED for each of the ceil(T/P) pages of a T-token
 * sequence into kinds[0..cap).  Returns the page count, or -1 on bad
 * arguments or when cap is too small.
 */
int32_t puzzlekv_classify_pages(int32_t T, int32_t P, int32_t sink_tokens, int32_t recent_tokens,
                                int32_t *kinds, int32_t cap);

/* Storage of one factorized key-value page pair relative to dense,
 * (r_K + r_V)(P + d) / (2 P d) [PuzzleKV §3.3 eq. (3)]. Host-only. */
double puzzlekv_page_storage_ratio(int32_t P, int32_t d, int32_t rank_k, int32_t rank_v);

/* Message of the calling thread's most recent failure ("" if none). */
const char *puzzlekv_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PUZZLEKV_H */
