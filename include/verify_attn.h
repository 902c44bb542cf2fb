/*
 * verify_attn.h -- C ABI of libverify_attn.so: speculative-decoding
 * verification attention on GB300 (sm_103a).
 *
 * T draft tokens of each sequence (a chain, a token tree given by parent
 * pointers, or a masked draft block) attend to the sequence's committed KV
 * cache and, under a bitmask, to one another.  The library computes it the
 * divide-and-aggregate way of LongSpec (section 2.C, "Hybrid Tree Attention"):
 * an unmasked split-KV pass over the cached prefix, a masked pass over the
 * draft block, and an exact log-sum-exp merge of the partial results.  The
 * prefix can be a contiguous cache, a paged cache behind a block table
 * (HiSpec, section 2, batched inference with paged attention), or a
 * fixed-size verify index set inside the full cache (Dustin, sections 1 and 3).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Pointers.  Every tensor argument is a DEVICE pointer to memory the caller
 *   allocated and owns; the library never allocates, frees or keeps a pointer
 *   after the call returns.  Only `shape` and the scalar arguments live on the
 *   host.  `workspace` is caller-owned device scratch of at least
 *   verify_attn_workspace_size() bytes, 256-byte aligned, initialised once with
 *   verify_attn_workspace_init() and reusable by later calls on the same stream,
 *   of this shape or of any other shape it is large enough for (its bookkeeping
 *   sits at fixed offsets and every completed call returns it to zero).  After
 *   a call that stopped at a bounded wait (verify_attn_check_status returns
 *   VA_ERR_TIMEOUT) run verify_attn_workspace_init() again before reusing it.
 *   Calls that run concurrently (different streams) need separate workspaces.
 * Streams.  Every call only enqueues work on `stream` (NULL = legacy default
 *   stream) and returns; nothing synchronises except verify_attn_check_status.
 * Layouts (row-major, contiguous unless a stride is given):
 *   q, out       [B][T][Hq][D]        element type shape->dtype
 *   lse          [B][Hq][T]           fp32, natural logarithm
 *   dense cache  [B][max_cache_len][Hkv][D]
 *   pages        [num_pages][page_size][Hkv][D]
 *   seqlens      [B] int32            committed prefix length L_b of sequence b
 *   tree_parent  [B][T] int32         -1 for a root, else 0 <= parent[i] < i
 *   tree_mask    [B][T][W] uint32     W = ceil(T/32); bit j%32 of word j/32 of
 *                                     row i set = draft token i sees draft token j
 *   positions    [B][T] int32         position id of draft token t (NULL = q and
 *                                     the draft keys already rotated; see
 *                                     "Rotary embedding" below)
 * Draft keys.  The T draft tokens' keys and values are already in the cache at
 *   logical slots L_b .. L_b+T-1 (append, then verify; rejected entries are
 *   dropped afterwards).
 * Rotary embedding (LongSpec section 1: the target keeps its own RoPE base;
 *   position ids may be arbitrary, e.g. anchor-offset ids).  With positions ==
 *   NULL the attention calls take q and the draft keys as stored (already
 *   rotated, e.g. by verify_rope_draft_*).  With positions != NULL they rotate
 *   q and the T draft keys on the fly, inside the attention kernels, exactly
 *   as verify_rope_draft_* would (rotate-half layout, element i with i + D/2,
 *   angle positions[b][t] * rope_base^(-2i/D), reduced modulo 2 pi to ~5e-7
 *   rad), and write neither q nor the cache; the prefix keys are taken as
 *   stored.  Requires shape->rope_base > 0 and |positions| < 2^24 (a larger
 *   one is recorded as VA_ERR_DEVICE_BOUNDS and taken as 0).  The accepted
 *   draft keys stay unrotated in the cache: once verify_commit_kv_* has moved
 *   them to L_b .. L_b+a-1, verify_rope_draft_* at the accepted tokens'
 *   positions rotates them for the next step (for a tree, L_b + depth).
 * GQA.  Query head h reads kv head h / (Hq/Hkv).
 * Draft visibility.  Exactly one of tree_parent / tree_mask may be non-NULL.
 *   With tree_parent, token i sees itself and its ancestors (computed inside
 *   the attention kernel).  With tree_mask, the bits decide.  With both NULL,
 *   the draft block is causal (a chain).  Every draft token sees the whole
 *   prefix (the cache part carries no mask).
 * Rows with no visible key (only possible with L_b = 0 and an empty mask row)
 *   get out = 0 and lse = -inf.
 * Errors.  A call returns VA_OK or an error code and never aborts.  Argument
 *   errors are found on the host before anything is enqueued.  Values that
 *   only the device can see (a seqlen beyond the cache, a page-table entry or
 *   verify index out of range, a bounded wait that ran out) are recorded in a
 *   status word inside the workspace; the kernel clamps or skips the bad value
 *   and finishes, so the output is then undefined but no fault occurs.
 *   verify_attn_check_status() reads and clears that word.
 *   verify_attn_last_error() describes the last error of the calling thread.
 */
#ifndef VERIFY_ATTN_H
#define VERIFY_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *va_stream; /* same type as cudaStream_t */

typedef enum {
  VA_OK = 0,
  VA_ERR_INVALID_ARG = 1,   /* bad pointer, size or combination of arguments */
  VA_ERR_UNSUPPORTED = 2,   /* valid but outside what this build supports */
  VA_ERR_WORKSPACE = 3,     /* workspace missing, misaligned or too small */
  VA_ERR_CUDA = 4,          /* a CUDA runtime call failed */
  VA_ERR_TIMEOUT = 5,       /* device: a bounded wait ran out */
  VA_ERR_DEVICE_BOUNDS = 6, /* device: seqlen / page / index out of range */
  VA_ERR_DEVICE_INVALID = 7 /* device, validation mode: a verify set that is not strictly increasing */
} va_status;

typedef enum { VA_DTYPE_BF16 = 0, VA_DTYPE_FP32 = 2 } va_dtype;

typedef enum { VA_LAYOUT_DENSE = 0, VA_LAYOUT_PAGED = 1, VA_LAYOUT_SPARSE = 2 } va_layout;

/* Problem shape.  Supported: 1 <= T <= 64; Hq % Hkv == 0; bf16 with D in
 * {64, 128}; fp32 with D = 64; B * Hkv * ceil(Hq/Hkv*T / 64) <= 2048. */
typedef struct {
  int B;         /* sequences in the batch */
  int T;         /* draft tokens per sequence */
  int Hq;        /* query heads */
  int Hkv;       /* key/value heads */
  int D;         /* head dimension */
  va_dtype dtype;/* element type of q, k, v and out */
  float scale;   /* score scale (1/sqrt(D) for standard attention) */
  float rope_base; /* RoPE base of the model, read only when an attention call
                    * is given positions (see "Rotary embedding" below) */
} va_shape;

/* Bytes of workspace the attention calls need for `shape` on the CURRENT
 * device (it depends on the device's SM count).  0 on invalid shape. */
size_t verify_attn_workspace_size(const va_shape *shape);

/* Initialise a workspace: status word and merge bookkeeping (on `stream`).
 * Zeroes all ws_bytes; call once after allocating a workspace. */
va_status verify_attn_workspace_init(void *workspace, size_t ws_bytes, va_stream stream);

/*
 * Verification attention over a dense contiguous cache.
 * LongSpec section 2.C: unmasked split-KV pass over the L_b cached keys
 * (FlashAttention-style, no mask), masked pass over the T draft keys at slots
 * L_b..L_b+T-1, exact log-sum-exp merge.  Requires L_b + T <= max_cache_len
 * (checked on the device).  positions: NULL, or [B][T] int32 position ids
 * of the draft tokens to rotate q and the draft keys on the fly (see "Rotary
 * embedding" above; verify_rope_draft_* is the separate pass).
 */
va_status verify_attn_dense(const va_shape *shape, const void *q, const void *k_cache,
                            const void *v_cache, int max_cache_len, const int32_t *seqlens,
                            const int32_t *tree_parent, const uint32_t *tree_mask,
                            const int32_t *positions, void *out, float *lse, void *workspace,
                            size_t ws_bytes, va_stream stream);

/*
 * verify_attn_dense for callers that cannot allocate device memory: the same
 * computation and arguments, but no workspace.  Meant for code that is handed
 * only its input and output buffers (for example a plugin inside a host
 * framework that owns the device allocator) and for deployments that fix their
 * device memory at start-up and allow no allocation afterwards.  The papers
 * have no counterpart: this is an interface convenience, not part of the method.
 *
 * Scratch.  The partial results, segment bookkeeping and status word live in
 * one file-scope device array of 8 MiB that every GPU which loads this library
 * holds until the process exits.  The first call on a device looks up that
 * array's device address (cudaGetSymbolAddress, with the device current); make
 * that first call before any stream capture.  No call allocates or frees
 * memory.  A shape whose scratch exceeds 8 MiB (verify_attn_workspace_size) is
 * rejected with VA_ERR_UNSUPPORTED before anything is enqueued.  On a 152-SM
 * GPU, d 128 and at most 32 packed query rows per kv-head (GQA group x T),
 * about 350 (sequence, kv-head) pairs fit -- e.g. one sequence with 8 draft
 * tokens, or 16 sequences of 5; a batch of 64 sequences of 16 does not.
 * Sharing.  Every call uses the same array and leaves its contents behind;
 * each call first clears the array's bookkeeping (status word and merge
 * counters, 16.6 KB), so a call is unaffected by the shape or the outcome of
 * the one before it.  Calls whose work overlaps on the
 * GPU (different streams, or different host threads) race on the array and
 * give undefined results: serialise them.
 * device_status (may be NULL): a caller-owned device int32 that receives this
 * call's device status word (VA_OK or the first device-side error), copied on
 * `stream` after the computation.
 */
va_status verify_attn_dense_noalloc(const va_shape *shape, const void *q, const void *k_cache,
                                    const void *v_cache, int max_cache_len, const int32_t *seqlens,
                                    const int32_t *tree_parent, const uint32_t *tree_mask,
                                    const int32_t *positions, void *out, float *lse,
                                    int32_t *device_status, va_stream stream);

/*
 * Verification attention over a paged cache (HiSpec section 2: paged attention
 * with block tables, so each sequence of a batch can accept a different
 * number of tokens without padding).  Logical slot p of sequence b lives at
 * page page_table[b][p / page_size], row p % page_size.  The draft keys are
 * logical slots L_b..L_b+T-1.  Requires L_b + T <= max_pages_per_seq *
 * page_size and 0 <= page < num_pages for every page read (device-checked).
 * page_size must be a power of two between 1 and 1024.
 */
va_status verify_attn_paged(const va_shape *shape, const void *q, const void *k_pages,
                            const void *v_pages, int num_pages, int page_size,
                            const int32_t *page_table, int max_pages_per_seq,
                            const int32_t *seqlens, const int32_t *tree_parent,
                            const uint32_t *tree_mask, const int32_t *positions, void *out,
                            float *lse, void *workspace, size_t ws_bytes, va_stream stream);

/*
 * Sparse verification (Dustin sections 1 and 3): the prefix part attends only
 * to the cache rows listed in the verify set of its (sequence, kv-head); the
 * cache itself is not compacted.  indices [B][Hkv][max_indices] int32 with
 * n_indices [B][Hkv] valid entries each, every entry in [0, L_b) (device
 * checked); order does not matter for the result, but a verify set is a set:
 * an index listed twice is attended twice.  The draft block is always read
 * from the dense slots L_b..L_b+T-1 under the draft mask.
 * Validation mode: with the environment variable VA_DEBUG_VALIDATE=1 the call
 * first checks every row on the device -- n_indices in [0, max_indices] and
 * its entries strictly increasing inside [0, L_b), the form verify_build_index
 * writes -- and records VA_ERR_DEVICE_INVALID for a row with an entry out of
 * order or listed twice (VA_ERR_DEVICE_BOUNDS for one out of range).
 */
va_status verify_attn_sparse(const va_shape *shape, const void *q, const void *k_cache,
                             const void *v_cache, int max_cache_len, const int32_t *seqlens,
                             const int32_t *indices, const int32_t *n_indices, int max_indices,
                             const int32_t *tree_parent, const uint32_t *tree_mask,
                             const int32_t *positions, void *out, float *lse, void *workspace,
                             size_t ws_bytes, va_stream stream);

/*
 * Exact log-sum-exp merge of partial attentions of the same rows (LongSpec
 * 2.C, the log-sum-exp fusion): lse = ln sum_s exp(lse_s), out = sum_s
 * exp(lse_s - lse) * o_s.  o_parts [n_parts][n_rows][D] fp32 (each part
 * normalised over its own keys), lse_parts [n_parts][n_rows] fp32 natural
 * log (-inf = empty part) -> out [n_rows][D] of out_dtype, lse [n_rows] fp32
 * (lse may be NULL).  Exposed for merging parts computed elsewhere, e.g. by
 * other ranks of a context-parallel split.  D in {64, 128}, n_parts <= 1024,
 * o_parts 16-byte aligned (VA_ERR_INVALID_ARG otherwise).
 */
va_status verify_attn_combine(int n_rows, int n_parts, int D, const float *o_parts,
                              const float *lse_parts, va_dtype out_dtype, void *out, float *lse,
                              va_stream stream);

/*
 * Ancestor-or-self bitmask of token trees (LongSpec 1.3 and 2.C: every branch
 * of the speculation tree attends to its own path).  parent [B][T] int32 as
 * above -> mask [B][T][ceil(T/32)] uint32.  1 <= T <= 64.  A parent entry
 * that breaks -1 <= parent[i] < i is recorded as VA_ERR_DEVICE_BOUNDS in the
 * status word of `workspace` (which may be NULL to skip recording) and its
 * row is cut at that node.
 */
va_status verify_tree_mask_from_parents(int B, int T, const int32_t *parent, uint32_t *mask,
                                        void *workspace, va_stream stream);

/*
 * Fixed-size verify index set (Dustin section 1, hybrid attention
 * aggregation), per (sequence b, kv-head h) with L = seqlens[b]:
 *   I = {0..n_sink-1} U {L-window..L-1}
 *       U top-m_draft positions of score_draft among the other positions
 *       U the highest score_target positions among those still unchosen,
 *         until |I| = min(budget, L),
 * clipped to [0, L), written sorted ascending to indices[b][h][0..n) with the
 * tail of the row set to -1, and n to n_indices[b][h].  Equal scores are
 * taken in increasing position order; -0.0 and +0.0 count as equal; scores
 * must not be NaN.  score_* are fp32 [B][Hkv][score_stride].  Requires
 * budget >= n_sink + window, L <= score_stride and L <= 131072 (a longer L is
 * recorded as VA_ERR_DEVICE_BOUNDS and clamped).  `workspace` (may be NULL)
 * receives device-side errors.
 */
va_status verify_build_index(int B, int Hkv, const int32_t *seqlens, const float *score_draft,
                             const float *score_target, int score_stride, int n_sink, int window,
                             int m_draft, int budget, int32_t *indices, int32_t *n_indices,
                             void *workspace, va_stream stream);

/*
 * Rotary position embedding of the draft block, in place (LongSpec section 1:
 * the target model keeps its own RoPE base; position ids may be arbitrary,
 * e.g. the anchor-offset ids 0, 1, 2, 3, 8192, 8193, ...).  For every
 * sequence b and draft token t < T, with p = positions[b][t]:
 *   every query head of q[b][t], and the key row of every kv-head at logical
 *   slot L_b + t of the cache (L_b = seqlens[b]),
 * are rotated pairwise in the rotate-half layout: element i pairs with
 * element i + D/2 (i < D/2) at the angle p * rope_base^(-2i/D),
 *   x'[i] = x[i] cos - x[i+D/2] sin,   x'[i+D/2] = x[i+D/2] cos + x[i] sin.
 * Angles are formed and reduced in fp64, rows rotated in fp32 and rounded
 * back to the element type.  Use: append the draft keys and values
 * unrotated at slots L_b .. L_b+T-1, call this with the draft tokens'
 * positions (L_b + depth for a tree, so an accepted path ends up rotated as
 * a plain sequence after verify_commit_kv_*), then call verify_attn_*.  The
 * value cache and every other key row are not touched.
 *   shape: B, T (<= 64), Hq, Hkv (<= 256), D (even, <= 256), dtype bf16 or
 *     fp32; scale is not used.
 *   q [B][T][Hq][D], positions [B][T] int32 (any value), seqlens [B] int32.
 *   Dense: k_cache [B][max_cache_len][Hkv][D], L_b + T <= max_cache_len.
 *   Paged: k_pages [num_pages][page_size][Hkv][D] behind page_table as for
 *     verify_attn_paged.
 * A sequence whose L_b or page entries are out of range keeps its key rows
 * unrotated (its q rows are still rotated) and VA_ERR_DEVICE_BOUNDS is
 * recorded in `workspace` (may be NULL).
 */
va_status verify_rope_draft_dense(const va_shape *shape, void *q, void *k_cache, int max_cache_len,
                                  const int32_t *seqlens, const int32_t *positions, float rope_base,
                                  void *workspace, va_stream stream);

va_status verify_rope_draft_paged(const va_shape *shape, void *q, void *k_pages, int num_pages,
                                  int page_size, const int32_t *page_table, int max_pages_per_seq,
                                  const int32_t *seqlens, const int32_t *positions, float rope_base,
                                  void *workspace, va_stream stream);

/*
 * Importance of the committed positions from a few query heads, the signal
 * that feeds verify_build_index (Dustin section 1: the target model's
 * attention scores are one signal of the global importance map; section 2:
 * the estimate is computed on a few semantic retrieval heads only).  For
 * sequence b with L = seqlens[b], every listed query head h and every token
 * t < T of q, p[h,t] is the attention distribution of q[b][t][h] over the L
 * committed keys of kv-head h / (Hq/Hkv) (score scale shape->scale; the rows
 * after the prefix take no part), and
 *   score[b][g][j] = sum over the listed heads and the T tokens of p[h,t][j]
 * for j < L and every kv-head g: one map per sequence, repeated in each
 * kv-head row so that verify_build_index takes it unchanged.  Entries
 * j >= L are not written.
 *   shape: B, T (<= 64), Hq, Hkv, scale; bf16 with D = 128 only.
 *   q [B][T][Hq][128] and k_cache [B][max_cache_len][Hkv][128] bf16, 16-byte
 *     aligned; seqlens [B] int32 (L <= max_cache_len and L <= score_stride,
 *     device-checked: a bad value is recorded and clamped).
 *   heads: HOST array of n_heads query-head indices in [0, Hq), 1 <= n_heads
 *     <= 32, n_heads * T <= 256; a head listed twice counts twice.
 *   score fp32 [B][Hkv][score_stride], 4-byte aligned.
 *   scratch: caller-owned device memory of at least
 *     verify_head_importance_scratch_size() bytes, 256-byte aligned (scores
 *     of the listed heads and per-chunk partial sums; contents not kept).
 *   workspace (may be NULL) receives device-side errors.
 * Two kernels on `stream`; calls that share a scratch buffer must not overlap.
 */
size_t verify_head_importance_scratch_size(int B, int T, int n_heads, int max_cache_len);

va_status verify_head_importance(const va_shape *shape, const void *q, const void *k_cache,
                                 int max_cache_len, const int32_t *seqlens, const int32_t *heads,
                                 int n_heads, float *score, int score_stride, void *scratch,
                                 size_t scratch_bytes, void *workspace, va_stream stream);

/*
 * After verification (Dustin section 1, step 5: accepted tokens join the
 * cache, rejected ones are dropped; HiSpec section 2: the entries of rejected
 * tokens are removed before the next phase, and the output equals the target
 * model's own decoding).
 *
 * Greedy acceptance over token trees.  parent [B][T] int32 as for the
 * attention calls; draft_tokens [B][T] int32; target_next [B][T+1] int32:
 * column 0 is the target model's greedy next token after the committed
 * prefix, column t+1 the one after draft node t.  A node is accepted when its
 * parent is accepted (or it is a child of the prefix, parent -1) and its token
 * equals the target's token after that parent.  Outputs, all device int32:
 * path [B][T] -- the deepest accepted root path as node indices from the root
 * down (the one ending at the smallest node index when several are equally
 * deep), tail -1; n_accept [B] -- its length (0 when no node is accepted);
 * bonus [B] -- the target's token after the path's last node (column 0 when
 * nothing is accepted).  1 <= T <= 64.  A parent entry that breaks
 * -1 <= parent[i] < i is recorded as VA_ERR_DEVICE_BOUNDS in the status word
 * of `workspace` (may be NULL) and that node counts as rejected.
 */
va_status verify_accept_greedy(int B, int T, const int32_t *parent, const int32_t *draft_tokens,
                               const int32_t *target_next, int32_t *path, int32_t *n_accept, int32_t *bonus,
                               void *workspace, va_stream stream);

/*
 * KV commit after acceptance, in place.  The draft rows of sequence b sit at
 * logical slots L_b .. L_b+T-1 (L_b = seqlens[b]); for j < n_accept[b] the
 * row at slot L_b + path[b][j] is moved to slot L_b + j, in every kv-head of
 * both caches.  Other slots keep their rows (those past L_b + n_accept[b]
 * are free for the next step).  path and n_accept as returned by
 * verify_accept_greedy: path[b][j] in [j, T).  seqlens_out [B] (may be NULL,
 * must not alias seqlens) receives L_b + n_accept[b].  shape supplies B, T
 * (<= 64), Hkv, D and dtype (Hq and scale are not used); rows of D elements
 * must be a multiple of 16 bytes.  Dense: caches [B][max_cache_len][Hkv][D],
 * L_b + T <= max_cache_len.  Paged: pages [num_pages][page_size][Hkv][D]
 * behind page_table [B][max_pages_per_seq] as for verify_attn_paged.  Caches
 * 16-byte aligned.  A seqlen, n_accept, path entry or page entry out of range
 * is recorded as VA_ERR_DEVICE_BOUNDS in `workspace` (may be NULL); the rows
 * it concerns are left in place.
 */
va_status verify_commit_kv_dense(const va_shape *shape, void *k_cache, void *v_cache, int max_cache_len,
                                 const int32_t *seqlens, const int32_t *path, const int32_t *n_accept,
                                 int32_t *seqlens_out, void *workspace, va_stream stream);
va_status verify_commit_kv_paged(const va_shape *shape, void *k_pages, void *v_pages, int num_pages,
                                 int page_size, const int32_t *page_table, int max_pages_per_seq,
                                 const int32_t *seqlens, const int32_t *path, const int32_t *n_accept,
                                 int32_t *seqlens_out, void *workspace, va_stream stream);

/* Wait for `stream`, read and clear the device status word of `workspace`.
 * Returns VA_OK or the first device-side error recorded since the last check.
 * After VA_ERR_TIMEOUT the workspace needs verify_attn_workspace_init() before
 * its next attention call (a merge counter may have been left mid-count). */
va_status verify_attn_check_status(void *workspace, va_stream stream);

/* Message for the last error returned on the calling thread ("" if none). */
const char *verify_attn_last_error(void);

/* Library version string, e.g. "verify_attn 0.1 sm_103a". */
const char *verify_attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* VERIFY_ATTN_H */
