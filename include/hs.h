/*
 * hs.h — C ABI of the Hybrid HiSparse sparse-MLA decode step on GB300 (sm_103a).
 *
 * What the library computes (sources are vLLM's Hybrid HiSparse write-ups):
 *   "Un contexte d'un million sur huit H200", section "Ce qui se passe":
 *     an indexer scores every cached token, the top-K are selected, and
 *     sparse MLA attention reads only those K latent rows; one indexer layer
 *     serves four sparse-MLA layers (IndexShare); the indexer cache stays
 *     resident on the GPU.
 *   same page, section "Les trois états de résidence":
 *     full residency (all rows on the GPU), mixed residency (the tail stays on
 *     the GPU and is never evicted, older pages live in pinned host memory,
 *     selected rows of them go to hot buffers), zero residency (nothing on the
 *     GPU; rows arrive as the indexer asks for them).  One fused resolve reads
 *     resident rows in place, refreshes the LRU entry of a hot row, and on a
 *     miss copies exactly one row from pinned host memory.  No CPU decision on
 *     the decode path, so the step can be captured in a CUDA graph.  Hot
 *     buffers are ordinary blocks of the same pool.
 *   same page, section "Ce qu'il faut en retenir":
 *     hot buffers hold 2 x top-K rows per request; with MTP,
 *     (num_speculative_tokens + 2) x top-K.
 *   "vLLM sert GLM-5.3 en contexte 1M sur 16 H200", section "Comment s'y
 *     prendre": top-K = 2048 selected tokens.
 *
 * Conventions for every function below:
 *   - Return value: HS_OK or an error status.  Argument errors are detected on
 *     the host before anything is enqueued; nothing is enqueued then.
 *   - Errors found on the device (an index outside the request, a hot buffer
 *     too small, a bounded wait that ran out) set a sticky device error word
 *     (read it with hs_pool_get_error); the affected kernel skips the work it
 *     cannot do and never traps.
 *   - "dev" pointers are CUDA device pointers owned by the caller; "host"
 *     pointers are host memory owned by the caller.  The library keeps no
 *     pointer to caller buffers beyond the call, except the two arenas given
 *     to hs_pool_create.
 *   - Hot-path calls (hs_indexer_score, hs_topk, hs_indexer_topk, hs_resolve,
 *     hs_sparse_mla_decode, hs_resolve_attend, hs_step) only enqueue work on
 *     `stream` (hs_resolve_attend and hs_step with a host pool also on the
 *     pool's side stream, joined back into `stream` by events before they
 *     return): no host synchronisation, no allocation, no branch on device
 *     data.  They may be
 *     captured in a CUDA graph and replayed.  What they launch depends only
 *     on the pool's configuration and the call's B and nq, so a captured
 *     graph stays valid when requests change residency or grow (hs_append)
 *     between replays.
 *   - A pool is not thread-safe; use it from one host thread and one stream
 *     at a time.
 *   - Batch index b of a hot-path call is request id b (0 <= b < B).  Calls
 *     that score, select or resolve tokens (hs_indexer_score, hs_topk,
 *     hs_indexer_topk, hs_resolve, hs_step) need every request to hold at
 *     least nq tokens (the step's own tokens are already in the cache):
 *     otherwise HS_ERR_INVALID_ARG and nothing is enqueued.
 */
#ifndef HS_H
#define HS_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    HS_OK = 0,
    HS_ERR_INVALID_ARG = 1,     /* bad argument, unknown request, wrong mode   */
    HS_ERR_ARENA_TOO_SMALL = 2, /* an arena is smaller than required           */
    HS_ERR_CAPACITY = 3,        /* no free GPU block / hot buffer too small     */
    HS_ERR_HOST_POOL_FULL = 4,  /* no free block in the pinned host pool        */
    HS_ERR_INDEX_RANGE = 5,     /* a selected index outside [0, seq_len)        */
    HS_ERR_TIMEOUT = 6,         /* a bounded device wait ran out                */
    HS_ERR_CUDA = 7,            /* a CUDA runtime call failed                   */
    HS_ERR_RANGE = 8            /* a value beyond the fp16 range of the tensor-core
                                   attention (a row's group scale s with
                                   448 * s > 65504, a query or rope value
                                   above 65504 in magnitude)               */
} hs_status;

/* Storage format of one MLA latent row (576 values = 512 nope + 64 rope). */
typedef enum {
    /* 656 bytes: [0,512) E4M3 codes of the nope dims, [512,528) four fp32
     * scales (one per 128 nope dims), [528,656) 64 bf16 rope dims. */
    HS_ROW_E4M3_656 = 0,
    /* 2304 bytes: 576 fp32 values. */
    HS_ROW_F32_2304 = 1
} hs_row_format;

/* Element format of indexer queries and keys. */
typedef enum { HS_IDX_E4M3 = 0, HS_IDX_F32 = 1 } hs_idx_format;

/* Residency of one request ("Les trois états de résidence"). */
typedef enum {
    HS_FULL = 0,  /* every page on the GPU                                   */
    HS_MIXED = 1, /* tail window on the GPU, older pages host-only, hot buffer */
    HS_ZERO = 2   /* nothing on the GPU, hot buffer filled on demand          */
} hs_mode;

typedef struct hs_pool hs_pool;

typedef struct {
    int32_t max_requests;   /* request ids are 0 .. max_requests-1              */
    int32_t max_tokens;     /* context capacity of one request                  */
    int32_t page_tokens;    /* P: tokens per page/block (64)                    */
    int32_t top_k;          /* K                                                */
    int32_t num_spec;       /* speculative tokens; nq = num_spec + 1 queries    */
    int32_t tail_tokens;    /* T: tail window kept on the GPU in mixed mode     */
    int32_t num_mla_layers; /* L: sparse-MLA layers served by one indexer layer */
    int32_t mla_heads;      /* H: attention heads of one MLA layer              */
    int32_t idx_heads;      /* Hi: indexer heads                                */
    int32_t idx_dim;        /* Di: indexer head dim                             */
    int32_t row_fmt;        /* hs_row_format                                    */
    int32_t idx_fmt;        /* hs_idx_format                                    */
    int32_t hot_rows;       /* C: hot-buffer rows per request; 0 selects the
                               pages' rule (num_spec + 2) * top_k.  Must be a
                               multiple of page_tokens and >= top_k.  Below
                               nq * top_k a step can find fewer free slots
                               than misses: hs_resolve then serves the lowest
                               missed tokens that fit, leaves the others
                               unread (row id -1) and reports HS_ERR_CAPACITY */
    int32_t reserved;
    int64_t gpu_blocks;     /* blocks in the device pool (each P tokens x L rows);
                               gpu_blocks * P <= 2^31 - 1 (row ids are int32) and
                               gpu_blocks * P * L < 2^32                        */
    int64_t host_blocks;    /* blocks in the pinned host pool (same shape); 0 =
                               no host copies (full residency only)            */
} hs_pool_config;

typedef struct {
    uint64_t resident; /* selected rows read in place (unique per request-step) */
    uint64_t hits;     /* hot-buffer hits                                      */
    uint64_t misses;   /* rows copied from pinned host (per request-step)      */
    uint64_t bytes_copied; /* misses x L x row bytes                           */
} hs_stats;

/* Byte offsets of the regions the pool carved from the device arena, for
 * inspection by tests and tools.  All offsets are from the arena base. */
typedef struct {
    size_t rows;             /* MLA block pool [gpu_blocks][L][P][R] bytes        */
    size_t idx_keys;         /* indexer keys [max_requests][max_tokens][Di] elems */
    size_t idx_scale;        /* indexer key scale [max_requests][max_tokens] fp32 */
    size_t block_table;      /* [max_requests][max_pages] int32, -1 = not on GPU  */
    size_t host_block_table; /* [max_requests][max_pages] int32, -1 = no host copy */
    size_t hot_map;          /* [max_requests][max_tokens] int32 slot or -1       */
    size_t slot_token;       /* [max_requests][C] int32 token or -1               */
    size_t stamp;            /* [max_requests][C] uint32 last-use step, 0 = never */
    size_t hot_blocks;       /* [max_requests][C/P] int32 pool block of each hot page */
    size_t seq_len;          /* [max_requests] int32                              */
    size_t req_step;         /* [max_requests] uint32 last resolved step          */
    size_t row_bytes;        /* R                                                 */
    size_t max_pages;        /* ceil(max_tokens / P)                              */
    size_t hot_rows;         /* C                                                 */
    size_t total;            /* bytes used of the arena                           */
} hs_layout;

/* ------------------------------------------------------------------------ */
/* Pool creation (host, off the decode path)                                 */
/* ------------------------------------------------------------------------ */

/* Bytes of device and pinned-host arena a pool with this config needs.
 * Pure host arithmetic; needs no GPU.  HS_ERR_INVALID_ARG for a bad config. */
hs_status hs_pool_required_bytes(const hs_pool_config *cfg, size_t *dev_bytes,
                                 size_t *host_bytes);

/* Carve a pool out of caller-owned memory: the shared block pool that holds
 * resident pages, tails and hot buffers alike, and the pinned host pool
 * ("Un contexte d'un million sur huit H200", « Les trois états de
 * résidence »; hot buffers of (num_spec + 2) * K rows: « Ce qu'il faut en
 * retenir »).  dev_arena: device memory of at
 * least *dev_bytes (16-byte aligned, 256 recommended).  host_arena: pinned
 * host memory (cudaHostAlloc / torch pin_memory) of at least *host_bytes, or
 * NULL when cfg->host_blocks == 0; it must be reachable from the device
 * (unified addressing).  Both must outlive the pool; the pool never allocates
 * device or pinned memory after this call.  Initialises the arena's tables
 * (synchronously on the default stream).  Errors: HS_ERR_INVALID_ARG (a bad
 * config, a NULL or unaligned arena, a host arena that is not pinned or not
 * reachable from the device), HS_ERR_ARENA_TOO_SMALL, HS_ERR_CUDA; *out is
 * then NULL and nothing the call made stays allocated (the arenas remain
 * the caller's). */
hs_status hs_pool_create(const hs_pool_config *cfg, void *dev_arena,
                         size_t dev_bytes, void *host_arena, size_t host_bytes,
                         hs_pool **out);
void hs_pool_destroy(hs_pool *pool);
hs_status hs_pool_get_layout(const hs_pool *pool, hs_layout *out);

/* ------------------------------------------------------------------------ */
/* Request lifecycle (host, between decode steps)                            */
/* ------------------------------------------------------------------------ */

/* Open request `req` (empty, length 0) in residency `mode`.  Mixed and zero
 * modes lease C/P hot-buffer blocks from the device pool and start with every
 * slot empty ("Les trois états de résidence": zero residency starts with empty
 * slots).  HS_ERR_CAPACITY when the pool lacks the blocks. */
hs_status hs_request_open(hs_pool *pool, int32_t req, hs_mode mode);

/* Append n tokens to request `req`.  mla_rows: [n][L][R] bytes; idx_keys:
 * [n][Di] elements of the indexer format; idx_scale: [n] fp32 (NULL = 1.0).
 * Each pointer may be host or device memory.  Rows of a page that is resident
 * (full mode: every page; mixed: the tail window) are written to the GPU pool
 * only; rows of a page that is not are written to the pinned host pool.  The
 * host copy of a resident page is left to hs_precopy ("Les trois états de
 * résidence": completed prefix pages are copied to the host ahead of time);
 * a page that slides out of the tail window (mixed mode) gets it here, on
 * `stream`, when no pre-copy has made it, and then gives its GPU block back.
 * With a host pool, every page also reserves its host block here.
 * Synchronises `stream` before returning (off the decode path); never waits
 * for pre-copies still in flight unless a page they cover leaves the GPU.
 * HS_ERR_CAPACITY: no GPU block; HS_ERR_HOST_POOL_FULL: no host block;
 * HS_ERR_INVALID_ARG: past max_tokens.  Nothing changes on these errors. */
hs_status hs_append(hs_pool *pool, int32_t req, const void *mla_rows,
                    const void *idx_keys, const float *idx_scale, int32_t n,
                    cudaStream_t stream);

/* Change the residency of a request between steps ("Les trois états de
 * résidence": full, mixed, zero), in any direction.  Pages that the new mode
 * keeps off the GPU (outside the tail window in mixed mode, all of them in
 * zero mode) release their GPU blocks, after their host copy is written on
 * `stream` (or `stream` is ordered after the pre-copy that wrote it); pages it
 * keeps on the GPU that are not there get a block and their rows copied back
 * from the host pool; a hot buffer is leased when leaving full residency and
 * returned when entering it; the hot buffer starts empty.  Needs a host pool
 * (HS_ERR_INVALID_ARG otherwise); HS_ERR_CAPACITY, with nothing changed, when
 * the pool lacks the blocks.  The pressure policy below stops managing the
 * request.  Synchronises `stream`. */
hs_status hs_request_set_mode(hs_pool *pool, int32_t req, hs_mode mode,
                              cudaStream_t stream);

/* Release every GPU and host block of the request (after any pre-copy still
 * in flight, which may touch them, has finished). */
hs_status hs_request_close(hs_pool *pool, int32_t req);

/* Pre-copy of completed pages ("Les trois états de résidence": in full
 * residency the completed prefix pages are copied to the host ahead of time,
 * so that they can later give their GPU slot up with no further copy).
 * Enqueues on `stream`, normally a side stream of the caller's, one
 * device->host copy per run of neighbouring blocks, covering every completed
 * page (all P tokens appended) of every open request that is on the GPU and
 * has no host copy yet.  The copies run on the copy engine, not the SMs, and
 * the call returns without waiting for them: decode steps go on meanwhile
 * (they only read those blocks).  Calls that later take one of those blocks
 * away (hs_append's tail roll-out, hs_request_set_mode, the pressure calls)
 * order their own stream after these copies on the device; hs_request_close
 * and hs_pool_destroy wait for them on the host.  Each call also orders
 * `stream` after the previous batch.  *pages (may be NULL): pages enqueued.
 * HS_ERR_INVALID_ARG without a host pool. */
hs_status hs_precopy(hs_pool *pool, cudaStream_t stream, int64_t *pages);

/* Pressure policy ("Ce qui se passe": the cache stays on the GPU while there
 * is room, and offloading applies only under real memory pressure; the pages
 * give no policy, so this is a reading).  Append as hs_append; when the
 * append does not fit in the free GPU blocks, flip to mixed residency the
 * full-residency request with the most resident pages among those whose flip
 * frees blocks (lower id on ties), and retry, until the append fits.  The
 * blocks a flip frees join the shared pool: the flipped request's own hot
 * buffer and any other request's next pages or hot buffer come out of it.
 * flipped: host [max_requests] (may be NULL) receives the flipped ids in
 * order, *n_flipped their number (flips stay done on error).
 * HS_ERR_CAPACITY when no flip is left that would free a block. */
hs_status hs_append_pressure(hs_pool *pool, int32_t req, const void *mla_rows,
                             const void *idx_keys, const float *idx_scale,
                             int32_t n, cudaStream_t stream, int32_t *flipped,
                             int32_t *n_flipped);

/* The other half of the pressure policy (reading): return requests that
 * hs_append_pressure flipped to full residency, the last flipped first, while
 * the free GPU blocks cover the pages that come back (less the hot buffer
 * given up) plus one block per open request (room for each one's next page,
 * so a return is not undone by the next appends).  Stops at the first that
 * does not fit.  restored: host [max_requests] (may be NULL), *n_restored
 * their number. */
hs_status hs_pool_relieve(hs_pool *pool, cudaStream_t stream, int32_t *restored,
                          int32_t *n_restored);

/* Number of free blocks left in the device pool. */
int64_t hs_pool_free_gpu_blocks(const hs_pool *pool);

/* ------------------------------------------------------------------------ */
/* Decode-step calls (async on `stream`, graph-capturable)                   */
/* ------------------------------------------------------------------------ */

/* Indexer score ("Ce qui se passe"): for b < B, query j < nq, token t <
 * seq_len[b]:
 *   scores[(b*nq + j)*score_stride + t] =
 *       sum_h w[b][j][h] * ReLU(sigma[b][t] * (q[b][j][h][:] . k[b][t][:]))
 * with ReLU(x) = x > 0 ? x : +0 (fp32).  q: dev [B][nq][Hi][Di] in the pool's
 * indexer format (E4M3 bytes or fp32); w: dev [B][nq][Hi] fp32; scores: dev
 * fp32, score_stride >= max_tokens.  Entries t >= seq_len[b] are untouched. */
hs_status hs_indexer_score(hs_pool *pool, const void *q, const float *w,
                           int32_t B, int32_t nq, float *scores,
                           int64_t score_stride, cudaStream_t stream);

/* Top-K ("Un contexte d'un million sur huit H200", « Ce qui se passe »: the
 * indexer picks the top-K tokens; K = 2048 selected tokens: "vLLM sert
 * GLM-5.3 en contexte 1M sur 16 H200", « Comment s'y prendre »): for each
 * (b, j) the K largest scores[(b*nq+j)*score_stride + t] over
 * t < seq_len[b] - nq + j + 1 (query j sees up to its own position); equal
 * scores go to the lower t; written ascending to topk[(b*nq+j)*K ..] and
 * padded with -1 when fewer than K tokens are visible.  Deterministic. */
hs_status hs_topk(hs_pool *pool, const float *scores, int64_t score_stride,
                  int32_t B, int32_t nq, int32_t *topk, cudaStream_t stream);

/* The same top-K as hs_topk for callers that cannot allocate device memory
 * and have no pool: for example a serving engine that reserved most of the
 * GPU for its own block pool at start-up (a later cudaMalloc would fail or
 * split that reservation), or host code that must avoid the device-wide
 * synchronisation of an allocation call.  The paper has no counterpart; this
 * is a library convenience.
 *   scores, score_stride, B, nq, K, topk: as for hs_topk (K = top_k);
 *   seq_len: dev [B] int32 request lengths (query j of request b sees
 *            t < seq_len[b] - nq + j + 1);
 *   max_tokens: tokens of each score row the call may read, <= score_stride;
 *            a query sees min(seq_len[b] - nq + j + 1, max_tokens) tokens, so
 *            a seq_len[b] beyond max_tokens is clamped on the device and no
 *            score past max_tokens is read.
 * Scratch: a static area inside this library (578 KiB of device memory,
 * held on every GPU that loads the library until the process exits).  Nothing is allocated or freed by this call.  Limits: B * nq <= 64
 * and max_tokens <= 1,048,576; larger requests return HS_ERR_CAPACITY and
 * enqueue nothing.  The first call on a device looks up the scratch's device
 * address (host-side set-up, once per device; make that first call before
 * any stream capture).  All calls share the one scratch area: each call
 * clears what must start at zero, but two calls whose kernels overlap on the
 * GPU (different streams, no ordering between them) race on it. */
hs_status hs_topk_noalloc(const float *scores, int64_t score_stride,
                          const int32_t *seq_len, int32_t B, int32_t nq,
                          int32_t K, int32_t max_tokens, int32_t *topk,
                          cudaStream_t stream);

/* hs_indexer_score + hs_topk with the scores kept in the pool's workspace
 * (« Ce qui se passe »: the indexer scores every cached token and picks the
 * top-K).  Errors as for those two calls. */
hs_status hs_indexer_topk(hs_pool *pool, const void *q, const float *w,
                          int32_t B, int32_t nq, int32_t *topk,
                          cudaStream_t stream);

/* Fused resolve ("Les trois états de résidence") of one step for requests
 * b < B.  topk: dev [B][nq][K] (ascending per (b,j), -1 padded).  Per request:
 * the union U of its nq lists; each u in U is resident (its page is on the
 * GPU: read in place), a hit (in the hot buffer: its stamp becomes this step,
 * i.e. the LRU entry is refreshed) or a miss.  Misses take the least recently
 * used slots not touched in this step (order (stamp, slot)); the i-th miss in
 * ascending token order takes the i-th such victim in ascending slot order;
 * then exactly one row per layer is copied from pinned host memory into the
 * slot.  row_id: dev [B][nq][K] int32, the pool row (block * P + offset) each
 * entry reads, -1 for padding.  The step number is a per-request device
 * counter incremented by this call (so graph replays keep counting).  With a
 * hot buffer below nq * K rows a request can have fewer slots not touched in
 * this step than misses: every such slot takes a miss (lowest tokens first),
 * the remaining misses get row id -1 (the attention skips them) and
 * HS_ERR_CAPACITY is set in the sticky error word. */
hs_status hs_resolve(hs_pool *pool, const int32_t *topk, int32_t B, int32_t nq,
                     int32_t *row_id, cudaStream_t stream);

/* The two halves of hs_resolve (« Les trois états de résidence »), for
 * callers that time them apart or run the
 * copy on another stream (ordered after the plan by an event):
 * hs_resolve_plan does the union, classification, LRU update and row ids,
 * and leaves the step's miss lists in the pool's workspace; hs_miss_copy then
 * copies exactly one row per miss and layer from pinned host memory into its
 * hot-buffer slot.  hs_miss_copy must follow the plan it copies for, with the
 * same B and nq, before the next plan; the rows of the misses are only there
 * once it has run.  hs_resolve = hs_resolve_plan + hs_miss_copy. */
hs_status hs_resolve_plan(hs_pool *pool, const int32_t *topk, int32_t B, int32_t nq,
                          int32_t *row_id, cudaStream_t stream);
hs_status hs_miss_copy(hs_pool *pool, int32_t B, int32_t nq, cudaStream_t stream);

/* The copy of hs_miss_copy for layers [layer_begin, layer_end) only, on a
 * grid of about `ctas` CTAs in all (0: about four per SM over the batch, as
 * hs_miss_copy).  The copy itself is the one "Un contexte d'un million sur
 * huit H200", « Les trois états de résidence », defines: exactly one row
 * per miss and layer from pinned host memory into the request's hot buffer.  For callers that overlap each layer's copy with another
 * layer's attention on a second stream, as hs_resolve_attend does with
 * about 64 CTAs: the copy of layer l must complete before layer l's
 * hs_sparse_mla_decode reads the rows.  The same ordering rule as
 * hs_miss_copy holds: after the plan it copies for, before the next plan.
 * HS_ERR_INVALID_ARG for an empty or out-of-range layer range, ctas < 0
 * or a batch the pool cannot hold; without a host pool there is nothing to
 * copy and the call returns HS_OK. */
hs_status hs_miss_copy_layers(hs_pool *pool, int32_t B, int32_t nq, int32_t layer_begin,
                              int32_t layer_end, int32_t ctas, cudaStream_t stream);

/* Timing of the per-layer miss copies (« Les trois états de résidence »)
 * that hs_resolve_attend and hs_step run on the pool's side stream: an
 * instrument for the step's host-link rate, no part of the method.  With enable != 0, every later such call
 * records a pair of pool-owned timing events around each layer's copy on
 * that stream (recorded as external events, so that a CUDA graph captured
 * after enabling keeps them and records them at every replay).
 * hs_pool_copy_times writes the durations, in ms, of layers [0, n) of the
 * last recorded step; call it once that step has completed (after a
 * stream or device synchronisation).  HS_ERR_INVALID_ARG without a host
 * pool or for n outside [0, L]; HS_ERR_CUDA when the events have not been
 * recorded or have not completed. */
hs_status hs_pool_time_copies(hs_pool *pool, int32_t enable);
hs_status hs_pool_copy_times(hs_pool *pool, float *ms, int32_t n);

/* Sparse MLA decode of one layer over the resolved rows ("Ce qui se passe"):
 *   z[b][j][h][k] = softmax_scale * q[b][j][h][:576] . row(row_id[b][j][k])[:576]
 *   out[b][j][h][:512] = sum_k softmax_k(z) * row[:512]   (rows with id -1 skipped)
 *   lse[b][j][h] = ln(sum_k exp(z))                        (if lse != NULL)
 * q: dev [B][nq][H][576] bf16; out: dev [B][nq][H][512] bf16; lse: dev fp32
 * or NULL.  q and out are read and written in 16-byte vectors: both must be
 * 16-byte aligned (HS_ERR_INVALID_ARG otherwise).  A query with no row gets
 * out = 0, lse = -inf.  With E4M3 rows and a head count that is a multiple of
 * 64, the products run on the tensor cores with fp16 operands (queries and
 * dequantised rows converted, fp32 accumulation): their magnitudes must stay
 * below 65504.  A row whose group scale s has 448 * s > 65504, or a query or
 * rope value beyond 65504 in magnitude, sets HS_ERR_RANGE in the sticky error
 * word (the output of that query is then not meaningful). */
hs_status hs_sparse_mla_decode(hs_pool *pool, int32_t layer, const void *q,
                               const int32_t *row_id, int32_t B, int32_t nq,
                               float softmax_scale, void *out, float *lse,
                               cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Token-partitioned decode on one GPU ("vLLM sert GLM-5.3 en contexte 1M sur */
/* 16 H200", « Le mécanisme »: decode context parallelism spreads the KV cache */
/* over the GPUs by tokens and gathers the fragments at every layer; here the  */
/* global top-K is taken over the shards' candidates and the shards' attention */
/* partials are merged by their log-sum-exp).  A request's                     */
/* R shards are R pool requests holding consecutive token ranges; with rows =  */
/* B * nq, shard r of row i is row r * rows + i of the batched calls.          */
/* ------------------------------------------------------------------------ */

/* Global top-K from the shards' local top-K lists.  scores: dev fp32 as written
 * by hs_indexer_score for the R*B shard requests, [R][rows][score_stride];
 * local_topk: dev [R][rows][K] (hs_topk of the shards: local token indices,
 * ascending, -1 padded); offsets: dev [R] int32, ascending first global token
 * of each shard.  Writes topk: dev [rows][K], the K best candidates by score
 * (equal scores: lower global token first) as global tokens, ascending, -1
 * padded: exactly hs_topk over the unsharded row, since every token of the
 * global top-K is in its shard's top-K; and part_topk: dev [R][rows][K], each
 * shard's entries of that list as local indices (ascending, -1 padded), the
 * lists its hs_resolve / hs_sparse_mla_decode take.  K = the pool's top_k,
 * R <= 8, R * K <= 16384 (HS_ERR_CAPACITY beyond, nothing enqueued). */
hs_status hs_dcp_topk_merge(hs_pool *pool, const float *scores, int64_t score_stride,
                            const int32_t *local_topk, const int32_t *offsets, int32_t R,
                            int32_t rows, int32_t *topk, int32_t *part_topk,
                            cudaStream_t stream);

/* Merge the shards' attention outputs (decode context parallelism: "vLLM
 * sert GLM-5.3 en contexte 1M sur 16 H200", « Le mécanisme »): o_parts dev
 * [R][rows][H][512] bf16 and
 * lse_parts dev [R][rows][H] fp32 (hs_sparse_mla_decode of each shard over
 * its part_topk rows) -> out dev [rows][H][512] bf16 = sum_r w_r o_r with
 * w_r = exp(lse_r - lse), lse = ln sum_r exp(lse_r) (written if lse != NULL).
 * A shard without rows (lse -inf) weighs nothing.  R <= 8. */
hs_status hs_dcp_combine(const void *o_parts, const float *lse_parts, int32_t R, int32_t rows,
                         int32_t H, void *out, float *lse, cudaStream_t stream);

/* Resolve + the sparse MLA decode of every layer of the group (« Les trois
 * états de résidence »; attention over the selected rows only: « Ce qui se
 * passe »), for a top-K
 * the caller already has (the second half of hs_step, e.g. for a selection
 * made elsewhere): the results of hs_resolve followed by hs_sparse_mla_decode
 * for each of the L layers.  Without a host pool everything is enqueued on
 * `stream`.  With one, the plan and the attentions go on `stream` and layer
 * l's missed rows are copied on a side stream the pool owns (about 64 CTAs
 * at the highest stream priority), so that layer l's copy runs while layer
 * l-1 attends; `stream` waits for each layer's copy by an event just before
 * that layer's attention, so when `stream` reaches the end of this call all
 * of the call's work is done (a CUDA graph captured on `stream` takes the
 * side stream's work in with it).  topk, row_id: as for hs_resolve; q_mla,
 * out, lse: as in hs_step_args ([L][B][nq]...). */
hs_status hs_resolve_attend(hs_pool *pool, const int32_t *topk, int32_t B, int32_t nq,
                            const void *q_mla, float softmax_scale, void *out, float *lse,
                            int32_t *row_id, cudaStream_t stream);

typedef struct {
    int32_t B, nq;
    const void *q_idx;    /* dev [B][nq][Hi][Di], indexer format             */
    const float *w_idx;   /* dev [B][nq][Hi]                                 */
    const void *q_mla;    /* dev [L][B][nq][H][576] bf16, 16-byte aligned    */
    float softmax_scale;
    void *out;            /* dev [L][B][nq][H][512] bf16, 16-byte aligned    */
    float *lse;           /* dev [L][B][nq][H] fp32, or NULL                 */
    int32_t *topk;        /* dev [B][nq][K] int32 (output)                   */
    int32_t *row_id;      /* dev [B][nq][K] int32 (output)                   */
    const int32_t *topk_in; /* dev [B][nq][K] int32, or NULL: lists for the  */
                            /* resolve in place of the indexer's top-K (which */
                            /* is still computed and written to topk)         */
} hs_step_args;

/* One decode step of one IndexShare group ("Un contexte d'un million sur
 * huit H200", « Ce qui se passe »: one indexer layer serves four sparse-MLA
 * layers): indexer score -> top-K ->
 * fused resolve (with miss copies) -> sparse MLA decode for each of the L
 * layers, i.e. the indexer's top-K followed by hs_resolve_attend (of
 * topk_in when it is given).  Enqueued on `stream`; no host
 * synchronisation. */
hs_status hs_step(hs_pool *pool, const hs_step_args *args, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Introspection (host, synchronising)                                       */
/* ------------------------------------------------------------------------ */

/* Synchronise the device, read and clear the sticky device error word. */
hs_status hs_pool_get_error(hs_pool *pool, hs_status *device_status);

/* Synchronise, read the device counters (cumulative since create/reset). */
hs_status hs_pool_stats(hs_pool *pool, hs_stats *out);
hs_status hs_pool_reset_stats(hs_pool *pool);

/* Copy one request's residency state to host arrays (any may be NULL):
 * hot_map [max_tokens], slot_token [C], stamp [C], block_table [max_pages],
 * host_block_table [max_pages], hot_blocks [C/P], step (1), seq_len (1). */
hs_status hs_pool_dump_state(hs_pool *pool, int32_t req, int32_t *hot_map,
                             int32_t *slot_token, uint32_t *stamp,
                             int32_t *block_table, int32_t *host_block_table,
                             int32_t *hot_blocks, uint32_t *step,
                             int32_t *seq_len);

/* Overwrite one request's hot-buffer state (hot_map, slot_token, stamp, step)
 * from host arrays, e.g. to re-seed a benchmark step.  The rows of the slots
 * are not touched. */
hs_status hs_pool_load_state(hs_pool *pool, int32_t req, const int32_t *hot_map,
                             const int32_t *slot_token, const uint32_t *stamp,
                             uint32_t step);

/* Number of kernels hs_step enqueues for a batch of B requests x nq queries,
 * those on the pool's side stream included (host arithmetic, the same
 * decision hs_step makes); -1 on bad arguments. */
int32_t hs_step_kernel_count(const hs_pool *pool, int32_t B, int32_t nq);

/* Failure-path check: enqueue on `stream` one small kernel that waits, with
 * the same bounded routine every hot-path kernel uses, on an mbarrier that
 * nothing completes, for limit_cycles SM cycles (1e3 .. 2e9).  The wait runs
 * out, HS_ERR_TIMEOUT lands in the pool's sticky error word (read and
 * cleared by hs_pool_get_error) and the context stays usable.  The pages
 * have no counterpart; it exists so that the timeout path can be tested
 * without faulting or hanging a GPU.  HS_ERR_INVALID_ARG for a limit out of
 * range. */
hs_status hs_check_wait_timeout(hs_pool *pool, int64_t limit_cycles, cudaStream_t stream);

/* Host-link probe: copy `bytes` of pinned host memory (host_src, allocated
 * with cudaHostAlloc / torch pin_memory) into device memory (dev_dst) with a
 * kernel that reads the host memory through its device mapping, 16-byte
 * loads, four in flight per thread, `ctas` CTAs of 256 threads (0 = four per
 * SM): the same zero-copy reads as the miss copy, for measuring the rate the
 * host link gives them.  Both pointers 16-byte aligned, bytes a multiple of
 * 16.  Async on `stream`.  The pages have no counterpart; it exists so that
 * miss traffic can be reported against the link's measured rate. */
hs_status hs_host_read_probe(const void *host_src, void *dev_dst, size_t bytes, int32_t ctas,
                             cudaStream_t stream);

/* A static English description of a status. */
const char *hs_status_string(hs_status s);

/* Version of this ABI (major * 100 + minor). */
int32_t hs_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* HS_H */
