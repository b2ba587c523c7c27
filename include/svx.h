/*
 * svx.h - C ABI of the chunked multi-query verification-attention library.
 *
 * One verification round of speculative decoding ("Resource-Efficient
 * Speculative Decoding for Long-Context LLM Serving", section 4.2 "KV
 * Streaming for Multi-Query Verification"): the k+1 verification queries of
 * every request in a Cohort attend to
 *   - the committed KV history [0, C_b) (Sealed History, section 4.1 Eq. 4),
 *     pushed chunk by chunk; a chunk in pinned host memory is copied to HBM by
 *     the library's copy engine, a chunk already in device memory is used in
 *     place; every chunk serves all queries of the round, and
 *   - the GPU-resident candidate region (Speculative Frontier) under a causal
 *     or token-tree mask,
 * and the partial results are merged by online softmax, Eqs. (7)-(8), so the
 * output is full attention, Eqs. (6) and (9).
 *
 * Conventions
 *   bf16   IEEE bfloat16 (as torch.bfloat16), element-contiguous.
 *   B      requests in the round (Cohort), Hq / Hkv query / KV heads,
 *          G = Hq / Hkv (query head h uses KV head h / G), d head dimension,
 *          nq verification queries per request (k+1, or token-tree nodes).
 *   Query j of request b sits at absolute position C_b + j; candidate j is
 *   the KV of that position.  Query j always sees all history, itself and
 *   (chain) candidates 0..j-1 or (tree) its ancestors.
 *
 * Ownership: the caller owns Q, the history KV (host or device), the
 * candidate KV, O and LSE; the library owns its staging slots, fp32 state
 * workspace, events and any stream it creates.  Pinned host history must stay
 * unmodified until svx_round_finish's work has completed on the compute
 * stream.  Device buffers given to a round must stay valid until then too.
 *
 * Errors: every call returns an svx_status; svx_last_error() gives a
 * human-readable message for the last failing call on that context.  No call
 * throws, aborts or exits.  After SVX_ERR_CUDA from a failed CUDA call the
 * context should be destroyed; the report of a kernel's expired bounded wait
 * (svx_round_finish), or in the bounds-checked library of a skipped access, is
 * the exception, and the context runs on.
 *
 * Threads: a context is used by one host thread at a time.
 *
 * CUDA graphs: a round whose parts are all device memory or zero-copy host memory enqueues work on
 * the compute stream only, so svx_round_begin .. svx_round_finish (timeout_ms = 0) may be captured
 * into a CUDA graph on that stream and replayed; each replay computes the round on the captured
 * buffers' current contents.  Capture after one eager round (kernel set-up happens on first use).
 * Rounds that stage pinned host parts through the copy engine wait on events recorded by earlier
 * rounds and cannot be captured.
 */
#ifndef SVX_H
#define SVX_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SVX_OK = 0,
  SVX_ERR_INVALID_ARG = 1, /* bad pointer, size, range, layout or coverage */
  SVX_ERR_BAD_STATE = 2,   /* call out of begin -> {push|candidates}* -> finish order */
  SVX_ERR_OOM = 3,         /* device or pinned allocation failed in svx_create */
  SVX_ERR_CUDA = 4,        /* a CUDA runtime call failed (message has the CUDA error) */
  SVX_ERR_TIMEOUT = 5,     /* svx_round_finish: work not complete within timeout_ms */
  SVX_ERR_UNSUPPORTED = 6  /* shape outside what the kernels implement */
} svx_status;

typedef struct svx_ctx_s* svx_ctx;

/* svx_config.flags */
#define SVX_FLAG_TIMING 1u           /* record CUDA events around copies and kernels (svx_round_stats) */
#define SVX_FLAG_NO_TENSOR_CORES 2u  /* run the history chunk kernel on FP32 FMA instead of tcgen05 */
#define SVX_FLAG_ZERO_COPY 4u        /* read pinned host parts in place over the host link (no staging copy);
                                        the chunk kernel then runs at link speed on zero_copy_ctas SMs.
                                        A round's pushes (host and device parts) launch together at
                                        svx_round_finish, a request's consecutive chunks merged into one
                                        part (see SVX_FLAG_ADAPTIVE below) */
#define SVX_FLAG_ADAPTIVE 8u         /* per round, stage pinned host parts through the copy engine or read
                                        them in place (as SVX_FLAG_ZERO_COPY), whichever was measured
                                        faster: see below */

/* Context configuration.  Shapes are fixed for the context's lifetime (the
 * Cohort compatibility rule of section 4.2: one layer shape, verification
 * width bound, dtype, Hkv, d and chunk size per batched kernel). */
typedef struct {
  int32_t max_req;          /* >= 1, <= 256: requests per round */
  int32_t n_q_heads;        /* Hq, a multiple of n_kv_heads */
  int32_t n_kv_heads;       /* Hkv >= 1 */
  int32_t head_dim;         /* d: 64 or 128 */
  int32_t max_query;        /* 1..32: verification queries (= candidates) per request */
  int32_t max_chunk_tokens; /* >= 1: capacity of one request's part in a staging slot */
  int32_t n_slots;          /* 2 or 3 staging slots (double / triple buffering) */
  int32_t device;           /* CUDA device ordinal */
  void* compute_stream;     /* cudaStream_t for kernels; NULL: library creates one (highest priority) */
  void* copy_stream;        /* cudaStream_t for H2D chunk copies; NULL: library creates one */
  uint32_t flags;           /* SVX_FLAG_* */
  int32_t zero_copy_ctas;   /* with SVX_FLAG_ZERO_COPY: CTA budget (one CTA per SM) of a launch that
                               reads host parts; 0 = all SMs.  A tensor-core launch uses
                               max(1, budget / groups) CTAs for each of its groups (one per KV head
                               and pass of up to 64 query rows).  Fewer leave SMs free for
                               co-running work; on GB300, 8 CTAs already fill the host link. */
  int32_t staged_ctas;      /* CTA budget of chunk launches over parts the copy engine staged; 0 = all
                               SMs.  Such a launch only has to keep up with the host link, so a few
                               SMs suffice, and a smaller launch starts sooner beside co-running
                               work (a Draft model on the other SMs, section 4.3). */
} svx_config;

/* One request's contiguous slice of committed history, [tok_start, tok_start + n_tok).
 * k, v: bf16 [n_tok][Hkv][d], 16-byte aligned.  Pinned host memory (cudaHostAlloc or
 * cudaHostRegister) is staged through a slot by the copy engine (n_tok <= max_chunk_tokens), or,
 * with SVX_FLAG_ZERO_COPY, read in place by the chunk kernel over the host link (any n_tok);
 * device memory is read in place (any n_tok).  Pageable host memory is rejected. */
typedef struct {
  int32_t req;
  int32_t n_tok;
  int64_t tok_start;
  const void* k;
  const void* v;
} svx_part;

/* Adaptive streaming (SVX_FLAG_ADAPTIVE).  How fast the copy engine reads pinned host memory can depend
 * on the host: on GB300 hosts some pinned buffers were read at 5-150 GB/s by the copy engine while SM
 * loads of the same buffers (SVX_FLAG_ZERO_COPY on 32 SMs) held the ~210 GB/s of the host link, and the
 * copy engine slowed by half beside a co-running GEMM while in-place reads did not.  With this flag the
 * context times its pushes' transfers (CUDA events around each push's copies, or around the chunk
 * kernels of a round read in place; read without waiting once they have completed) and keeps each
 * engine's recent ms per GB (decayed sums of time and bytes over about the last 500 samples).  The engine
 * is chosen per round, when it begins, so no round mixes them.  A round read in place launches its parts
 * when svx_round_finish is called: a request's parts that continue one another (next tokens, next rows of
 * the same buffer) merge into one, and a launch holds at most one part per request, so pushing chunk by
 * chunk costs one launch per round as a rule; the timing window counts those launches as one push.
 * Choice:
 * round 0 is staged and round 1 read in place (each engine measured once); after that, rounds are
 * staged through the copy engine unless in-place reads on zero_copy_ctas SMs were measured 10% faster
 * per byte (and then read in place until the copy engine is measured 5% faster than them), and one whole round
 * uses the other engine after 8 rounds, then 16, 32, ... up to 1024
 * while the preference holds (back to 8 when it changes), so a change of either rate is followed.
 * Results do not depend on the choice (both paths run the same arithmetic); only the transfer engine
 * changes. */

/* The adaptive policy's current figures: each engine's recent ms per GB of host history (-1 before its
 * first completed measurement) and whether it now prefers in-place reads.  Host-only; no waiting.
 * SVX_ERR_BAD_STATE without SVX_FLAG_ADAPTIVE. */
svx_status svx_adaptive_state(svx_ctx ctx, double* ce_ms_per_gb, double* ip_ms_per_gb, int32_t* prefer_in_place);

/* Allocates n_slots staging slots of max_req * max_chunk_tokens * Hkv * d * 2 bf16 each, the
 * fp32 (m, l, a) workspace and events on cfg->device.  Returns SVX_ERR_OOM, _INVALID_ARG,
 * _UNSUPPORTED or _CUDA on failure (then *out is NULL). */
svx_status svx_create(const svx_config* cfg, svx_ctx* out);

/* Waits for the context's outstanding work, then frees everything it owns.  NULL is a no-op. */
svx_status svx_destroy(svx_ctx ctx);

/* Starts a round (one layer of one Cohort).  q_dev: device bf16 [n_req][Hq][n_query][d].
 * hist_len_host: host int64[n_req], C_b >= 0.  scale: softmax scale; 0 means 1/sqrt(d)
 * (Eq. 6).  Running states start at (-inf, 0, 0) (section 4.2, online softmax). */
svx_status svx_round_begin(svx_ctx ctx, int32_t n_req, int32_t n_query, const void* q_dev,
                           const int64_t* hist_len_host, float scale);

/* Processes one Cohort chunk: at most one part per request.  Host parts are copied into the next
 * staging slot on the copy stream (waiting until the compute stream has released that slot);
 * the chunk kernel then updates every query's (m, l, a) with Eqs. (7)-(8).  Asynchronous: returns
 * once the work is enqueued.  Parts may arrive in any order across calls (the result does not
 * depend on chunk order, Eq. 9); svx_round_finish checks that they tile each [0, C_b) exactly once. */
svx_status svx_push_chunk(svx_ctx ctx, const svx_part* parts, int32_t n_parts);

/* The GPU-resident candidate region of the round (section 4.2, the causal mask by absolute
 * position).  k_dev, v_dev: device bf16 [n_req][n_cand][Hkv][d] with n_cand == n_query; they must
 * stay valid until the round's finish work has run.  parent_host: NULL for the causal chain
 * (query j sees candidates 0..j), else host int32[n_req][n_cand] token-tree parents with
 * parent[0] = -1 and 0 <= parent[i] < i (query j sees j and its ancestors); copied by this call.
 * The attention over the region is computed by svx_round_finish's kernel (one launch fewer per
 * round), so this call only validates and records.  At most once per round, in any order with
 * the pushes. */
svx_status svx_candidate_attn(svx_ctx ctx, const void* k_dev, const void* v_dev, int32_t n_cand,
                              const int32_t* parent_host);

/* Ends the round: checks chunk coverage, attends over the candidate region if one was given,
 * merges it with the history states (Eq. 8) and writes
 * O = a / l (Eq. 9) as bf16 [n_req][Hq][n_query][d] and LSE = m + ln l as fp32
 * [n_req][Hq][n_query] (natural log of the softmax denominator of the scaled scores) to device
 * memory.  A query with no visible key gets O = 0 and LSE = -inf.  timeout_ms = 0 returns
 * after enqueueing; > 0 waits on the host up to that long and returns SVX_ERR_TIMEOUT if the
 * work has not completed (the work stays enqueued), or SVX_ERR_CUDA if a kernel's bounded wait
 * gave up (2 s) in this round or in any round since the last finish with timeout_ms > 0: the
 * context's device error word keeps an expiry until such a finish reads it, reports it and clears
 * it.  The outputs of the round whose kernel gave up are invalid.  The context is ready for the
 * next round either way; its work is stream-ordered after this round's.  In the bounds-checked
 * library (libsvx_checked.so, built with -DSVX_BOUNDS_CHECK; the pages have no counterpart) every
 * kernel also checks that its global reads and writes lie in the buffers its launch describes, skips
 * one that does not and raises the same word (bit 4, and bit 8 + the site), which this call then
 * reports the same way. */
svx_status svx_round_finish(svx_ctx ctx, void* o_dev, float* lse_dev, int32_t timeout_ms);

/* Test hook of the failure path (the pages have no counterpart).  Enqueues on the compute stream,
 * between rounds, a one-thread kernel whose bounded wait on a barrier that nothing completes runs
 * out after wait_ms (1..2000) and raises the device error word, as a chunk kernel's waits do when
 * their producer never delivers.  The next svx_round_finish with timeout_ms > 0 then returns
 * SVX_ERR_CUDA ("a kernel gave up waiting"), clears the word, and the context runs further rounds.
 * SVX_ERR_BAD_STATE inside a round. */
svx_status svx_debug_expire_wait(svx_ctx ctx, int32_t wait_ms);

/* Test hooks of the host-side failure and overlap paths (the pages have no counterpart); they make a
 * failure on the host, never on the GPU.  Copy submissions are counted from the arming call (1 = the
 * next one the context issues); nth = 0 disarms.
 * svx_debug_fail_copy: the nth submission is refused as if cudaMemcpyAsync / cudaMemcpy2DAsync had
 * failed.  The push that meets it returns SVX_ERR_CUDA without launching its chunk kernel: copies it had
 * already issued are joined back into the copy stream, its parts do not count as pushed, and the round
 * stays open, so pushing the same chunk again completes it.  A failure of the CUDA call itself takes
 * the same path.
 * svx_debug_delay_copy: the host sleeps delay_ms (0..10000) before the nth submission.  A push's copy
 * interval starts at its first submission, so a pause before a push's first copy shows as copy-stream
 * idle time (copy_gap_ms, and chunk_kernel_exposed_ms for a chunk kernel that runs in it), and a pause
 * between two copies of a push lies inside that push's copy interval (a slow copy).
 * A 2D copy that the runtime refuses (its rows lie in different allocations; the parts are then copied
 * one by one) counts as a submission too. */
svx_status svx_debug_fail_copy(svx_ctx ctx, int64_t nth);
svx_status svx_debug_delay_copy(svx_ctx ctx, int64_t nth, int32_t delay_ms);

/* Test hook of the bounds-checked library (the pages have no counterpart).  From the next chunk launch
 * on, until svx_round_finish, the launches describe q as holding at most `rows` rows (rows < 0: the real
 * count again).  The real buffer is larger, so no access ever leaves it: in libsvx_checked.so the chunk
 * kernel skips its q loads past `rows` and raises the device error word, which svx_round_finish
 * (timeout_ms > 0) reports as SVX_ERR_CUDA; in libsvx.so the checks do not exist and the round is
 * unchanged.  It shows that the checked build's checks run and are reported. */
svx_status svx_debug_clip_q_rows(svx_ctx ctx, int64_t rows);

/* Message for the last failing call on ctx (never NULL; "" if none).  NULL ctx: last failure of
 * svx_create or svx_verify_static on this thread. */
const char* svx_last_error(svx_ctx ctx);

/* Per-round timing (needs SVX_FLAG_TIMING).  Waits for the last finished round to complete.  A round that
 * opens a new timing window (after svx_window_reset, or past a window's limits) reuses the window's
 * events, so the previous round's figures are no longer available from then on. */
typedef struct {
  double round_ms;        /* first event of the round to the end of its finish kernel */
  double copy_busy_ms;    /* sum over pushes of H2D copy time on the copy stream */
  double chunk_kernel_ms; /* sum over pushes of chunk-kernel time on the compute stream (from the
                             moment its staging slot is ready) */
  double cand_kernel_ms;  /* always 0: the candidate region runs inside the finish kernel */
  double finish_kernel_ms; /* candidate region + merge + finalize */
  int64_t h2d_bytes;      /* history bytes copied from host this round */
  int64_t device_bytes;   /* history bytes read in place from device memory this round */
  int32_t n_chunk_launches;
  int32_t n_copies;       /* host-to-device copy calls issued: two per host part, or two per chunk when
                             its host parts are equally strided rows of one batched tensor (2D copies) */
  double chunk_kernel_exposed_ms; /* time of chunk kernels that read staged or device parts, outside every
                                     transfer interval of the round (copies, and the kernels that read host
                                     parts in place); 1 - exposed / chunk_kernel_ms is the compute hidden
                                     under transfer */
  double transfer_busy_ms; /* length of the union of the transfer intervals */
  int32_t n_zero_copy_pushes; /* push intervals whose chunk kernels read host parts in place: a round read
                                 in place launches its pushes together and counts once */
} svx_stats;
svx_status svx_round_stats(svx_ctx ctx, svx_stats* out);

/* Timing over several rounds (needs SVX_FLAG_TIMING): the copy/compute timeline of a whole
 * multi-layer step, where layer l + 1's chunk copies overlap layer l's kernels (section 4.2,
 * "Pipelined KV transfers and prefetching").  A window opens at the first svx_round_begin after
 * svx_window_reset (or after svx_create) and takes every round up to the last finished one; it
 * holds at most 4096 rounds and 65536 pushes, and a round past either limit opens a new window.
 * Overlap within the window: copy_busy_ms sums the pushes' copy intervals on the copy stream
 * (slot released -> last copy of the push done), chunk_kernel_ms the chunk kernels' intervals on
 * the compute stream (from the moment the staging slot is ready), chunk_kernel_exposed_ms the
 * kernel time outside every copy interval, and copy_gap_ms the copy stream's idle time between its
 * first copy and its last.  1 - max(0, window_ms - copy_busy_ms) / (the same chunks' kernel time
 * with resident history) is the hidden fraction of compute over the whole step.  A round read in
 * place launches its pushes together at svx_round_finish: they form one push interval. */
typedef struct {
  double window_ms;        /* first round's begin (or the window's first copy, if that started earlier)
                              to the last finished round's finish-kernel end */
  double copy_busy_ms;
  double copy_gap_ms;
  double chunk_kernel_ms;
  double chunk_kernel_exposed_ms;
  double finish_kernel_ms; /* summed over the window's rounds */
  double transfer_busy_ms; /* union of copy intervals and in-place (zero-copy) chunk-kernel intervals */
  double zero_copy_kernel_ms; /* chunk-kernel time of pushes that read host parts in place */
  int32_t n_zero_copy_pushes;
  int32_t pad;
  int64_t h2d_bytes;       /* history bytes staged or read from host memory in the window */
  int64_t device_bytes;    /* history bytes read in place from device memory */
  int32_t n_rounds;
  int32_t n_pushes;
  int32_t n_chunk_launches;
  int32_t n_copies;
} svx_window_summary;
/* Opens a new window at the next svx_round_begin.  SVX_ERR_BAD_STATE inside a round. */
svx_status svx_window_reset(svx_ctx ctx);
/* Waits for the window's last finished round, then reports it.  SVX_ERR_BAD_STATE if none. */
svx_status svx_window_stats(svx_ctx ctx, svx_window_summary* out);
/* The window's pushes in issue order, 4 doubles each: copy start, copy end (both NaN for a push
 * without copies), chunk-kernel start, end; ms from the window's first round begin (a copy that the
 * copy stream started before the compute stream reached that event has a negative start).  Writes at most
 * cap pushes to out and the count to *n_out.  Waits like svx_window_stats. */
svx_status svx_window_intervals(svx_ctx ctx, double* out, int64_t cap, int64_t* n_out);
/* The window's rounds in order, 3 doubles each: round begin, finish-kernel start, finish-kernel end; ms
 * from the window's first round begin.  With svx_window_intervals this gives each round's (or each
 * step's) own length and transfer time.  Writes at most cap rounds; waits like svx_window_stats. */
svx_status svx_window_rounds(svx_ctx ctx, double* out, int64_t cap, int64_t* n_out);

/* ---- host-only bookkeeping (no GPU needed) ----------------------------------------------- */

/* One entry of a cohort chunk plan. */
typedef struct {
  int32_t chunk;     /* cohort chunk index j */
  int32_t slot;      /* staging slot j mod n_slots */
  int32_t req;
  int32_t n_tok;     /* min(chunk_tokens, C_b - tok_start) */
  int64_t tok_start; /* j * chunk_tokens */
} svx_plan_entry;

/* Cohort chunk plan (section 4.2, "Pipelined KV transfers" and "Cohort batching"): history of
 * each request cut into contiguous chunks of chunk_tokens; cohort chunk j holds one part per
 * request with C_b > j * chunk_tokens, in request order.  Writes at most cap entries to out and
 * the total count to *n_out (call with cap = 0 to size). */
svx_status svx_plan_chunks(int32_t n_req, const int64_t* hist_len, int32_t chunk_tokens, int32_t n_slots,
                           svx_plan_entry* out, int64_t cap, int64_t* n_out);

/* Candidate visibility words: out[b * n_query + j] bit i set iff query j of request b may
 * attend to candidate i.  parent NULL: chain (i <= j); else int32[n_req][n_query] tree
 * parents (i == j or i an ancestor of j).  n_query <= 32.  SVX_ERR_INVALID_ARG on a bad tree. */
svx_status svx_candidate_masks(int32_t n_req, int32_t n_query, const int32_t* parent, uint32_t* out);

/* Coverage check used by svx_round_finish: *ok_out = 1 iff the parts (req, tok_start, n_tok)
 * given as int64[n_parts][3] tile every [0, hist_len[b]) exactly once, else 0. */
svx_status svx_check_coverage(int32_t n_req, const int64_t* hist_len, const int64_t* parts, int64_t n_parts,
                              int32_t* ok_out);

/* Work plan of one tensor-core chunk launch (head_dim 128), as svx_push_chunk makes it; host only.
 * n_tok[n_parts] (1 <= n_parts <= 64): the parts' token counts; rows = G * n_query, the query rows
 * per KV head; cta_budget >= 1: CTAs available (the SM count, or zero_copy_ctas).  The grid is
 * n_groups = n_kv_heads * ceil(rows / rows_per_pass) CTA groups (one per KV head and pass of up to 64
 * rows) of ctas_per_group CTAs; a group walks the 128-token tiles of every part for its head and
 * pass, part after part (part i's first tile is tile_base[i] of tiles_per_group), and CTA j of a
 * group takes tiles [floor(j T / c), floor((j + 1) T / c)) with T = tiles_per_group and c =
 * ctas_per_group.  The grid shrinks until no part spans more than 8 CTAs (state slots); *slots is
 * the most it spans.  Out: *grid, *n_groups, *ctas_per_group, *tiles_per_group, *slots,
 * tile_base[n_parts].  SVX_ERR_INVALID_ARG on bad sizes or more than 2^31 - 1 tiles. */
svx_status svx_plan_tc(int32_t n_parts, const int32_t* n_tok, int32_t n_kv_heads, int32_t rows, int64_t cta_budget,
                       int64_t* grid, int32_t* n_groups, int32_t* ctas_per_group, int64_t* tiles_per_group,
                       int32_t* slots, int64_t* tile_base);

/* ---- a round that allocates nothing ------------------------------------------------------ */

/* Size of the library's static device scratch array (per GPU, held until the process exits). */
#define SVX_STATIC_SCRATCH_BYTES (32u << 20)

/* One whole verification round over device-resident KV without allocating any memory.  The paper
 * has no counterpart to this call: it exists for callers that cannot call cudaMalloc while they
 * run - an engine whose memory manager owns all device memory after start-up, or a decode loop
 * that cannot accept an allocation's cost or implicit synchronisation.  The fp32 (m, l, a)
 * state and an error word live in a static __device__ array of
 * SVX_STATIC_SCRATCH_BYTES that every GPU loading the library holds; the caller passes all
 * inputs and outputs.
 *
 * Computes what svx_round_begin + one in-place part per request + svx_candidate_attn +
 * svx_round_finish compute, on `stream` (cudaStream_t, NULL = default stream) of the calling
 * thread's current device, and returns once the work is enqueued.
 *   q_dev            bf16 [n_req][n_q_heads][n_query][head_dim]
 *   hist_len_host    int64[n_req], 0 <= C_b < 2^31
 *   k/v_hist_dev     host arrays of n_req device pointers, bf16 [C_b][n_kv_heads][head_dim]
 *                    (entries for C_b = 0 are ignored)
 *   k/v_cand_dev     bf16 [n_req][n_query][n_kv_heads][head_dim], or both NULL (no candidates)
 *   parent_host      NULL (causal chain) or int32[n_req][n_query] token-tree parents
 *   scale            0 means 1/sqrt(head_dim)
 *   o_dev, lse_dev   bf16 [n_req][n_q_heads][n_query][head_dim], fp32 [n_req][n_q_heads][n_query]
 * The state needs 8 * (16 + 4 * head_dim) bytes per query row (n_req * n_q_heads * n_query rows)
 * after a 256-byte header, so a call takes at most 7,943 query rows at head_dim 128 and 15,420 at
 * head_dim 64; larger rounds return SVX_ERR_INVALID_ARG and enqueue nothing.  The first call on a device sets up the scratch
 * (cudaGetSymbolAddress and a zeroing cudaMemset, synchronous); make that first call before any
 * stream capture.  All calls share the one array: calls whose GPU work overlaps (different
 * streams, or several host threads) race and give wrong results - order them on one stream.
 * Errors: SVX_ERR_INVALID_ARG, _UNSUPPORTED, _CUDA; message from svx_last_error(NULL). */
svx_status svx_verify_static(int32_t n_req, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                             int32_t n_query, const void* q_dev, const int64_t* hist_len_host,
                             const void* const* k_hist_dev, const void* const* v_hist_dev,
                             const void* k_cand_dev, const void* v_cand_dev, const int32_t* parent_host,
                             float scale, void* o_dev, float* lse_dev, void* stream);

/* Reads and clears the static scratch's device error word on the calling thread's current device:
 * *expired = 1 if a kernel of some svx_verify_static call since the last check gave up a bounded
 * wait (2 s; that call's outputs are invalid), or, in the bounds-checked library, skipped an access
 * outside its buffers, else 0.  Waits for all work on the device
 * (cudaDeviceSynchronize), so call it outside latency-critical loops and outside stream capture.
 * Allocates nothing.  Errors: SVX_ERR_INVALID_ARG, _CUDA; message from svx_last_error(NULL). */
svx_status svx_static_check(int32_t* expired);

/* ---- commit-aware KV tiering (host side of the history that the rounds stream) ------------- */

/* One request's Target KV regions (section 4.1, Eq. 4): Sealed History [0, H) in host memory,
 * Active Tail [H, C) and Speculative Frontier [C, L) on the GPU, 0 <= H <= C <= L.  Zero-initialise
 * with pending = -1.  `event` is owned by the library while a migration is in flight. */
typedef struct {
  int64_t H;        /* history confirmed in host memory */
  int64_t C;        /* committed prefix C_r */
  int64_t L;        /* logical length L_r, committed plus candidates */
  int64_t pending;  /* endpoint E of the migration in flight, or -1 */
  void* event;      /* CUDA event of that migration (library-owned), or NULL */
} svx_tier_state;

/* Eq. (5): E = max{H, g * floor(max(0, C - T) / g)}; T = Active Tail target, g = migration
 * granularity.  Needs g >= 1, T >= 0, 0 <= H <= C and H a multiple of g.  Host-only. */
svx_status svx_migration_endpoint(int64_t H, int64_t C, int64_t T, int64_t g, int64_t* E_out);

/* A new round: committed prefix C (never shrinks) and logical length L >= C.  Host-only. */
svx_status svx_tier_round(svx_tier_state* s, int64_t C, int64_t L);

/* Plans a migration with Eq. (5): if none is in flight and E > H, marks [H, E) pending and returns it
 * in [*begin, *end); otherwise *begin = *end = H.  Host-only (the caller copies). */
svx_status svx_tier_plan(svx_tier_state* s, int64_t T, int64_t g, int64_t* begin, int64_t* end);

/* The caller's copy of the pending interval has completed: H advances to its endpoint.
 * SVX_ERR_BAD_STATE while a copy enqueued by svx_tier_migrate is in flight (svx_tier_poll and
 * svx_tier_release advance H for those). */
svx_status svx_tier_complete(svx_tier_state* s);

/* End of round: keep the prefix [0, C_new), C <= C_new <= L, and release [C_new, L) on the GPU (the
 * released interval is returned).  It never meets [0, H) (SVX_ERR_BAD_STATE if it would). */
svx_status svx_tier_commit(svx_tier_state* s, int64_t C_new, int64_t* rel_begin, int64_t* rel_end);

/* Plans with Eq. (5) and, if E > H, enqueues on `stream` (cudaStream_t) the device-to-host copy of
 * rows [H, E) of K and V: k_dev_at_H / v_dev_at_H are the device addresses of position H, k_host /
 * v_host pinned host addresses of position 0 of the request's history; row_bytes = Hkv * d * 2.
 * H does not move until svx_tier_poll reports the copy complete (section 4.1).  *E_out = E (= H if
 * nothing moves).  SVX_ERR_BAD_STATE while a previous migration is still unpolled. */
svx_status svx_tier_migrate(svx_tier_state* s, int64_t T, int64_t g, int64_t row_bytes, const void* k_dev_at_H,
                            const void* v_dev_at_H, void* k_host, void* v_host, void* stream, int64_t* E_out);

/* *done = 1 and H advanced if the migration in flight has completed (or none was in flight), else 0. */
svx_status svx_tier_poll(svx_tier_state* s, int32_t* done);

/* Waits for a migration in flight, advances H and frees its event. */
svx_status svx_tier_release(svx_tier_state* s);

/* ---- Target-priority admission of Draft steps (host-side decisions) ------------------------ */

/* Section 4.3: a Draft step may start under the selected allocation only if the estimated Target
 * latency increase is within budget and the estimated Draft step time plus a margin fits the
 * remaining window; one step per request at a time; instructions expire; ACKs close steps; the
 * estimates follow observations (x <- x + ema * (observed - x)). */
typedef struct {
  double eps_target;    /* acceptable relative Target latency increase, eps_T >= 0 */
  double delta;         /* time margin for execution variability (same unit as all times) */
  double ema;           /* weight of the newest observation, (0, 1] */
  double t_draft;       /* offline Draft single-step time under the allocation, t_D(x, n0) */
  double delta_target;  /* offline relative Target latency increase under it, Delta_T(x, n0) */
  int32_t alloc;        /* the allocation n0 (e.g. TPCs or SMs given to the Draft) */
} svx_sched_config;

typedef struct svx_sched_s* svx_sched;

/* A scheduling instruction: t_latest = t0 + S_hat - t_D_hat - delta. */
typedef struct {
  int64_t req;
  int64_t round;
  int64_t seq;
  int32_t alloc;
  double t_latest;
} svx_draft_instr;

svx_status svx_sched_create(const svx_sched_config* cfg, svx_sched* out);
svx_status svx_sched_destroy(svx_sched s);
/* A new verification round: a pause ends once the latency estimate is back within budget. */
svx_status svx_sched_new_round(svx_sched s);
/* At time `now` with remaining window S_hat (`window`): *admitted = 1 and *out filled if a Draft step
 * for `req` may start, else 0 (paused, a step already unfinished, or a rule fails). */
svx_status svx_sched_try_admit(svx_sched s, int64_t req, int64_t round, double now, double window,
                               svx_draft_instr* out, int32_t* admitted);
/* Draft side, before starting: *ok = 1 iff the instruction matches the current request and round and
 * t_latest has not passed.  A rejected instruction is dropped (its request may be scheduled again). */
svx_status svx_sched_check_start(svx_sched s, const svx_draft_instr* ins, int64_t cur_req, int64_t cur_round,
                                 double now, int32_t* ok);
/* ACK of a finished step with its observed duration: *accepted = 1 if it closed the request's step. */
svx_status svx_sched_ack(svx_sched s, int64_t req, int64_t seq, double t_draft_observed, int32_t* accepted);
/* Observed Target latency with and without co-execution; over budget pauses new submissions. */
svx_status svx_sched_observe_target(svx_sched s, double t_co, double t_alone);
/* Current estimates t_D_hat, Delta_T_hat and the pause flag. */
svx_status svx_sched_estimates(svx_sched s, double* t_draft, double* delta_target, int32_t* paused);

/* ---- I/O-aware dynamic verification width (host-side controller) ---------------------------- */

/* Section 4.2: the next round's width is argmin over the candidate widths of the estimated round time
 * over the estimated committed tokens.  Round time = Draft generation + max(history transfer, attention)
 * + rejection correction (overlapped time counted once); every term and the committed count are moving
 * averages (weight ema on the newest round).  Each width is first tried n_init times, in the given
 * order; afterwards the width changes only if the best estimate beats the current width's by more than
 * `threshold` (relative); ties go to the earlier width. */
typedef struct svx_width_s* svx_width;
svx_status svx_width_create(const int32_t* widths, int32_t n, double ema, double threshold, int32_t n_init,
                            svx_width* out);
svx_status svx_width_destroy(svx_width w);
/* End-of-round statistics of a round verified at width q (q must be one of the widths). */
svx_status svx_width_record(svx_width w, int32_t q, double t_draft, double t_h2d, double t_attn, double t_correct,
                            double committed);
/* Width for the next round. */
svx_status svx_width_next(svx_width w, int32_t* q_out);
/* Current estimate T_round_hat(q) / U_hat(q), or -1 without records. */
svx_status svx_width_cost(svx_width w, int32_t q, double* cost_out);

/* Library version string. */
const char* svx_version(void);

/* sizeof of the ABI's structs, for bindings to check their layouts: svx_config, svx_part, svx_stats,
 * svx_window_summary, svx_plan_entry, svx_tier_state, svx_sched_config, svx_draft_instr, in this order.
 * Writes min(cap, count) entries to out and returns the count.  Host-only. */
int32_t svx_abi_sizes(int64_t* out, int32_t cap);

#ifdef __cplusplus
}
#endif

#endif /* SVX_H */
