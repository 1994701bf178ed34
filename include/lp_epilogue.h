/*
 * lp_epilogue.h -- C ABI of the GB300 (sm_103a) generation-logprob and greedy
 * speculative-acceptance epilogue.
 *
 * The operation (sources: "logprobs-design.md", the generation-logprob
 * captured-graph contract; "mtp-design.md", section "A speculative round is a
 * state transaction", steps 2-3):
 *
 *   Input is a block of target logits [rows, V_padded] (FP32 or BF16), split
 *   into verify groups.  Group g owns rows group_indptr[g] .. group_indptr[g+1]-1
 *   = [p, d0, ..., d(k-1)]: row j holds the target logits that check draft
 *   draft_tokens[row] (j < k); row k yields the bonus token.
 *
 *   1. Greedy acceptance.  a = number of leading rows j < k whose draft equals
 *      the row's argmax over raw logits (smallest id among equal maxima; -0 and
 *      +0 are one value).  The group emits rows 0..a: the chosen token of row
 *      j is its argmax (equal to the draft for j < a; the correction or bonus
 *      token for j = a).  A k = 0 group emits one row whose chosen token is
 *      sampled_tokens[g] when that is >= 0, else the argmax.  (mtp-design.md,
 *      same section, step 3: a accepted drafts yield a + 1 new tokens.)
 *   2. For every emitted row of a group whose requested[g] is nonzero:
 *      lse = log sum_v exp(logits[v]) over the V unpadded lanes, accumulated
 *      in FP32; lp(v) = fl32(logits[v] - lse), -0 reported as +0.
 *      (logprobs-design.md, opening paragraph: the logprob of token t is its
 *      logit minus the logsumexp of the whole vocabulary, summed in FP32.)
 *   3. The record of that row (258 int32 words):
 *        [0] chosen token id, [1] FP32 bits of its lp,
 *        [2+2i], [3+2i] = (id, lp bits) of alternative i:
 *          - id_counts[g] == 0: the top_k[g] (<= k_alt_max) natural
 *            alternatives, ordered by lp descending then id ascending, ties
 *            created by the FP32 subtraction included;
 *          - id_counts[g] = c > 0: token_ids[g][0..c) in caller order;
 *        every other pair = (-1, 0x7FC00000).
 *      (logprobs-design.md, packed-position paragraph: the chosen id and the
 *      bits of its FP32 logprob come first, then one (id, FP32 bits) pair per
 *      alternative, with -1 as the id of every unused pair.)
 *   4. Rows past a group's emitted prefix affect no output; a k = 0 group with
 *      requested[g] == 0 and sampled_tokens[g] >= 0 reads nothing.  Records of
 *      rows that are not emitted, or whose group is not requested, are not
 *      written.  By default such rows are not read either.  With
 *      LP_PLAN_READ_AHEAD, producers that would otherwise idle may read the
 *      row after a row still being decided, so that a verify chain can
 *      advance as soon as each decision is made; results are the same, and
 *      at most the first row past each prefix is read.
 *      (logprobs-design.md, the paragraphs on the speculative writer and on
 *      the request flag: positions past a request's committed prefix are left
 *      unread there, because in its packed layout they may belong to another
 *      request; a zero request flag skips the vocabulary pass, the sort and
 *      the record.  Here every row of the block belongs to its group, so a
 *      read-ahead read is safe.)
 *
 * Lifetime: lp_plan_create allocates all device scratch once; lp_bind records
 * caller-owned device pointers; lp_run only enqueues kernels on the caller's
 * stream (no allocation, no host synchronisation; capturable in a CUDA graph).
 * One plan serves one stream at a time; the plan must outlive queued work.
 * Binds and runs of one plan are not thread-safe.
 *
 * Residency: the stream kernel is persistent (a few CTAs per multiprocessor)
 * and its CTAs hand work to one another, but every work item is claimed
 * through a counter by a CTA that is already running, so a run does not need
 * the whole GPU: beside another kernel on another stream (or in a parallel
 * graph branch), the CTAs that are resident do all the work and the others,
 * when they start, find none.  The run then takes longer; it does not stall.
 * The records are built by a second persistent kernel while the stream
 * kernel runs; it is scheduled only once every stream CTA has started, takes
 * the room the stream kernel leaves, and waits on the stream kernel's
 * decisions, never the other way round.
 *
 * Errors: every function returns LP_OK (0) or a negative LP_E* code and never
 * aborts.  Conditions only visible on the device are reported in the bound
 * status word (LP_STATUS_* bits), which each lp_run resets to 0 first.
 */
#ifndef LP_EPILOGUE_H
#define LP_EPILOGUE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LP_RECORD_WORDS 258          /* chosen pair + 128 alternative pairs */
#define LP_MAX_IDS 128               /* explicit-id slots per group */
#define LP_MAX_K_ALT 32              /* largest natural-alternative count a plan accepts */
#define LP_MAX_DRAFTS 15             /* largest k (drafts per group) a plan accepts */
#define LP_UNUSED_LP_BITS 0x7FC00000u /* lp bits of an unused pair (a quiet NaN) */

/* Element type of the logit block. */
typedef enum { LP_F32 = 0, LP_BF16 = 1 } lp_dtype;

/* Host error codes. */
enum {
    LP_OK = 0,
    LP_EINVAL = -1,    /* NULL pointer or nonsensical argument */
    LP_ESHAPE = -2,    /* sizes inconsistent (V > V_padded, rows > max_rows, ...) */
    LP_EALIGN = -3,    /* logits not 16-byte aligned, or V_padded * elt not a multiple of 16 */
    LP_ECAPACITY = -4, /* request beyond the plan's limits (k_max, k_alt_max, max_ids) */
    LP_EDTYPE = -5,    /* unknown dtype */
    LP_ECUDA = -6,     /* a CUDA runtime call failed (see lp_last_cuda_error) */
    LP_ESTATE = -7,    /* lp_run before lp_bind, or host staging not enabled */
    LP_ESCRATCH = -8   /* lp_run_static: the run needs more scratch than its fixed array */
};

/* Device status bits (OR-ed into *status by a run). */
#define LP_STATUS_BAD_ID 0x1u    /* explicit id outside [0, V): pair = (id, 0x7FC00000) */
#define LP_STATUS_BAD_TOKEN 0x2u /* sampled token >= V: chosen lp bits = 0x7FC00000 */
#define LP_STATUS_BAD_COUNT 0x4u /* id count outside [0, max_ids] or top_k outside [0, k_alt_max]: clamped */
#define LP_STATUS_BAD_GROUP 0x8u /* group_indptr malformed: the run reads and writes nothing else */
#define LP_STATUS_TIMEOUT 0x10u  /* a bounded device wait expired: outputs are incomplete */
#define LP_STATUS_BAD_TEMPERATURE 0x20u /* lp_chain_verify: a temperature not in (0, inf): group skipped */

/* Plan flags. */
#define LP_PLAN_HOST_STAGING 0x1u     /* also allocate device staging so lp_run_host can be used */
#define LP_PLAN_READ_AHEAD 0x2u       /* idle producers may read the row after one being decided */
#define LP_PLAN_VOCAB_SHARDS 0x4u     /* also allocate the exchange buffers of lp_run_sharded */
#define LP_PLAN_DEBUG_FORCE_TIMEOUT 0x100u /* test hook: every bounded wait runs out (no reads) */
#define LP_PLAN_DEBUG_TRACE 0x200u    /* record a device timeline of each run (see lp_debug_trace) */

typedef struct {
    int32_t max_rows;     /* capacity: rows per run (>= 1) */
    int32_t max_groups;   /* capacity: groups per run (>= 1) */
    int32_t k_max;        /* largest drafts per group, 0..LP_MAX_DRAFTS */
    int64_t V;            /* unpadded vocabulary (>= 1) */
    int64_t V_padded;     /* row stride in elements (>= V) */
    int32_t dtype;        /* lp_dtype */
    int32_t k_alt_max;    /* largest top_k, 0..LP_MAX_K_ALT */
    int32_t max_ids;      /* largest id count, 0..LP_MAX_IDS */
    int32_t device;       /* CUDA device ordinal the plan lives on */
    uint32_t flags;       /* LP_PLAN_* */
    int64_t timeout_ns;   /* limit of every device-side wait, from kernel start; 0 = 1 s */
} lp_plan_desc;

/* Buffers of one run.  Device pointers for lp_bind, host pointers for
 * lp_run_host.  Layouts are dense row-major:
 *   logits         [rows, V_padded] of dtype   (input; lanes >= V are never used)
 *   group_indptr   int32 [groups + 1]          (0 <= indptr[0] < ... <= rows; sizes 1..k_max+1)
 *   draft_tokens   int32 [rows]                (row indptr[g]+j carries draft j of group g)
 *   sampled_tokens int32 [groups]              (k = 0 groups: chosen token; < 0 = argmax)
 *   requested      int32 [groups]              (nonzero = report logprobs)
 *   top_k          int32 [groups]              (natural alternatives, 0..k_alt_max)
 *   token_ids      int32 [groups, 128]         (explicit ids, caller order)
 *   id_counts      int32 [groups]              (0 = natural alternatives; 1..max_ids = explicit)
 *   records        int32 [rows, 258]           (output; only emitted rows of requested groups)
 *   accepted       int32 [groups]              (output: a, the accepted drafts)
 *   emitted_tokens int32 [rows]                (output: chosen token, -1 past the prefix)
 *   lse_out        float [rows] or NULL        (output: lse of rows whose record is written)
 *   status         uint32 [1]                  (output: LP_STATUS_* bits)
 */
typedef struct {
    const void* logits;
    const int32_t* group_indptr;
    const int32_t* draft_tokens;
    const int32_t* sampled_tokens;
    const int32_t* requested;
    const int32_t* top_k;
    const int32_t* token_ids;
    const int32_t* id_counts;
    int32_t* records;
    int32_t* accepted;
    int32_t* emitted_tokens;
    float* lse_out;
    uint32_t* status;
    int32_t rows;
    int32_t groups;
} lp_io;

typedef struct lp_plan_s* lp_plan_t;

/* Creates a plan on desc->device and allocates its device scratch (once).
 * Errors: LP_EINVAL, LP_ESHAPE, LP_EDTYPE, LP_ECAPACITY, LP_ECUDA. */
int lp_plan_create(lp_plan_t* out, const lp_plan_desc* desc);

/* Frees the plan's scratch.  The caller must have drained work queued with it. */
int lp_plan_destroy(lp_plan_t plan);

/* Device bytes lp_plan_create allocates for desc (0 if desc is invalid). */
size_t lp_plan_scratch_bytes(const lp_plan_desc* desc);

/* Validates and records the device buffers of the next runs.  Checks NULLs,
 * rows <= max_rows, groups <= max_groups, 16-byte alignment of logits and
 * 4-byte alignment of the int32 buffers.  Contents are validated on the
 * device (status bits).  Errors: LP_EINVAL, LP_ESHAPE, LP_EALIGN. */
int lp_bind(lp_plan_t plan, const lp_io* io);

/* ---- Commit clipping ("mtp-design.md", a speculative round, step 4 and the
 * paragraph after it)
 *
 * Attaches optional per-group clipping inputs to the bound buffers, for the
 * following lp_run calls (lp_bind clears them; lp_run_host, lp_run_static and
 * lp_score never clip).  Device pointers, or NULL for none:
 *   eos_tokens  int32 [groups]  the emitted prefix ends at the first emitted
 *                               token equal to it, which is kept (< 0 = none)
 *   budgets     int32 [groups]  at most this many tokens are emitted; <= 0 =
 *                               the request is at its limit and takes no step
 * With a accepted drafts the unclipped prefix holds a+1 tokens; the clipped
 * one holds t = min(a+1, budget, position of the first EOS + 1).  accepted[g]
 * then reports t - 1 and emitted_tokens holds -1 past the t tokens, so
 * records are written, and rows read, for the t emitted rows only.  A group
 * at its limit reports accepted -1, emits nothing and reads nothing.
 * Errors: LP_EINVAL (no plan), LP_ESTATE (nothing bound), LP_EALIGN. */
int lp_bind_clip(lp_plan_t plan, const int32_t* eos_tokens, const int32_t* budgets);

/* Enqueues the epilogue over the bound buffers on `stream` (a cudaStream_t;
 * NULL = legacy default stream).  Returns after enqueueing.  Errors:
 * LP_ESTATE (nothing bound), LP_ECUDA (launch failed). */
int lp_run(lp_plan_t plan, void* stream);

/* Same operation over HOST buffers (pinned for asynchronous copies): copies the
 * inputs and the output buffers (so that rows the run does not write keep the
 * caller's contents) to plan-owned device staging, runs, and copies records,
 * accepted, emitted_tokens, lse_out (if non-NULL) and status back, all on
 * `stream`.  When the logit block is pinned host memory mapped into the
 * device's address space (cudaHostAlloc'd or registered; 16-byte aligned), it
 * is not copied: the kernels read it in place, so only the rows the run reads
 * (and the gathered logits) cross the host link.
 * Returns after enqueueing; synchronise the stream before reading outputs.
 * Needs a plan created with LP_PLAN_HOST_STAGING (else LP_ESTATE).
 * Host buffers must stay valid until the stream reaches the end of the copies
 * (and, for logits read in place, until the run has completed). */
int lp_run_host(lp_plan_t plan, const lp_io* host_io, void* stream);

/* Bytes lp_run_host copies host->device and device->host for host_io.  Logits
 * read in place are not included: the run reads rows_read * V * element size
 * of them (rows_read from the accepted counts). */
int lp_run_host_bytes(lp_plan_t plan, const lp_io* host_io, int64_t* h2d, int64_t* d2h);

/* ---- Prompt scoring ("logprobs-design.md", the prompt-logprobs paragraphs)
 *
 * Scores target tokens against rows of logits: row j carries the logits that
 * predict target_tokens[j].  For a valid target t (0 <= t < V) the record holds
 *   [0] t, [1] FP32 bits of lp(t) = fl32(x_t - lse) (-0 reported as +0),
 *   [2] rank = 1 + the number of lanes v < V whose lp(v) is strictly greater,
 *   [3+2i], [4+2i] = (id, lp bits) of the 20 natural alternatives in the
 *       generation order (lp descending, id ascending), (-1, 0x7FC00000) past V;
 * for any other target (-1 marks the prompt end or an image position) the row
 * is not read and its record is id -1, 0x7FC00000, rank 0, every alternative
 * (-1, 0x7FC00000); a target >= V also sets LP_STATUS_BAD_TOKEN.  (The page:
 * each scored row holds the actual token id, its raw FP32 logprob bits, its
 * rank, then twenty alternatives; an invalid target row holds id -1, NaN,
 * rank zero and alternative ids -1.)
 *
 *   records      int32 [rows, 43]   (output; every row written)
 *   lse_out      float [rows] or NULL (output: lse of the rows read)
 *
 * The rank counts strictly greater *reported* values, so lanes whose logit is
 * above the target's but whose lp rounds to the same value do not count.
 * Uses the plan's scratch: rows <= max_rows and rows <= max_groups (each row
 * is scored on its own).  Device pointers; enqueues only, like lp_run.  The
 * bound lp_io buffers are neither used nor changed.
 * Errors: LP_EINVAL, LP_ESHAPE, LP_EALIGN, LP_ECUDA. */
#define LP_SCORE_WORDS 43
#define LP_SCORE_ALTS 20

typedef struct {
    const void* logits;            /* [rows, V_padded] of the plan's dtype, 16-byte aligned */
    const int32_t* target_tokens;  /* [rows] */
    int32_t* records;              /* [rows, 43] */
    float* lse_out;                /* [rows] or NULL */
    uint32_t* status;              /* [1] */
    int32_t rows;
} lp_score_io;

int lp_score(lp_plan_t plan, const lp_score_io* io, void* stream);

/* ---- Vocabulary-sharded records ----
 *
 * Source: "logprobs-design.md", the vocabulary-sharded speculative
 * verification paragraph.  Each rank holds a vocabulary shard of the target
 * logits.  A first exchange carries each shard's maximum and exponential mass
 * (the global normalisation); a second carries the chosen token's raw logit
 * from its owning rank and either the shard's best 32 sort keys or the selected
 * ids' raw logits, 256 words per position per rank; a final merge writes the
 * same packed record.
 *
 * lp_run_sharded runs the bound epilogue (as lp_run, same outputs) with the
 * records built that way over `shards` vocabulary shards of one block on one
 * GPU: shard s of a row is the column range of tiles [s*T/S, (s+1)*T/S) (T =
 * lp_plan_tiles_per_row).  Acceptance is decided first, as verification does
 * before the reduction.  Each shard's part touches only its own columns and
 * its own slot of two exchange buffers (plan memory, allocated at creation
 * with LP_PLAN_VOCAB_SHARDS: 8 + 1,024 bytes per row per shard for up to 8
 * shards); the gathers are the buffers read by the next launch.  Natural
 * alternatives are exact: each shard's 32 keys are its best 32 by (logprob
 * desc, id asc) under the global normalisation, so the merged K <= 32 are the
 * row's.  lse may differ from lp_run's in its last bit (another summation
 * order).  LP_ESTATE without LP_PLAN_VOCAB_SHARDS or a bind; LP_EINVAL unless
 * 1 <= shards <= min(8, T).  Enqueues only. */
int lp_run_sharded(lp_plan_t plan, int32_t shards, void* stream);

/* ---- Stochastic chain verification ----
 *
 * Source: "mtp-design.md", section "Sampling correctness".  A draft drawn
 * from the draft law q is accepted with probability min(1, p/q); at the first
 * rejection the next token is drawn from the positive residual max(p - q, 0),
 * normalised; after every draft is accepted the bonus token is drawn from the
 * target law of the bonus row.  For row j of group g (groups as in lp_bind:
 * rows r0..r0+k-1 carry drafts, row r0+k is the bonus row):
 *   p_j(v) = exp(x_j(v)/t - lse(x_j/t)) over the V unpadded lanes, t = temperature[g],
 *            with lse accumulated in FP32;
 *   draft j is accepted iff u[r0+j] * q_j(d_j) < p_j(d_j) (FP32), i.e. u < p/q;
 *   a = the number of leading accepted drafts;
 *   the last token is the smallest id v whose running sum of weights (ids in
 *   ascending order, FP64 sums of FP32 weights) exceeds r[g] times their
 *   total; the weights are max(p_a - q_a, 0) when a < k (p_a if that residual
 *   has no mass) and p_k when a == k.
 * The random numbers are inputs, so any generator (e.g. a counter-based
 * stream of the caller) can drive it.  Rows past a group's emitted prefix are
 * not read.  The plan's V, V_padded, dtype, k_max and device apply; its scratch
 * is not used.
 *
 *   logits        [rows, V_padded] of the plan's dtype (device)
 *   group_indptr  int32 [groups + 1]; group sizes 1..k_max + 1
 *   draft_tokens  int32 [rows]; row r0+j carries d_j (j < k)
 *   draft_probs   float [rows, V_padded]; row r0+j is q_j, the law that drew d_j
 *                 (16-byte aligned; rows r0+k are not read)
 *   temperature   float [groups] (> 0)
 *   u             float [rows] in [0, 1): acceptance uniforms of the draft rows
 *   r             float [groups] in [0, 1): the draw uniform of each group
 *   accepted      int32 [groups] (output: a; -1 for a skipped group)
 *   emitted       int32 [rows] (output: d_j for j < a, the drawn token at
 *                 j = a, -1 after)
 *   lse_out       float [rows] or NULL (output: lse(x_j/t) of every row read)
 *   status        uint32 [1] (output: reset, then LP_STATUS_* bits:
 *                 BAD_GROUP for a malformed group (skipped, accepted -1),
 *                 BAD_TEMPERATURE (skipped, accepted and emitted -1), BAD_TOKEN
 *                 for a draft >= V (rejected))
 * Host errors as for lp_bind (LP_EALIGN: logits or draft_probs not 16-byte
 * aligned).  Enqueues only; no allocation. */
typedef struct {
    const void* logits;
    const int32_t* group_indptr;
    const int32_t* draft_tokens;
    const float* draft_probs;
    const float* temperature;
    const float* u;
    const float* r;
    int32_t* accepted;
    int32_t* emitted;
    float* lse_out;
    uint32_t* status;
    int32_t rows;
    int32_t groups;
} lp_chain_io;

int lp_chain_verify(lp_plan_t plan, const lp_chain_io* io, void* stream);

/* Debug: number of vocabulary tiles the last run read for each row (0 = the
 * row was never read), copied into host_tiles[0..rows).  With
 * LP_PLAN_READ_AHEAD the first row past a prefix may show read-ahead tiles.  Synchronises the
 * plan's last stream.  A tile is 32 KiB of logits: 16384 BF16 or 8192 FP32
 * elements (the last tile of a row may be shorter). */
int lp_debug_tiles_read(lp_plan_t plan, int32_t* host_tiles, int32_t rows);

/* Debug: fills the plan's per-tile partial-result scratch with NaN bytes on
 * `stream` (to show that no result depends on stale scratch). */
int lp_debug_poison_scratch(lp_plan_t plan, void* stream);

/* Debug: the device timeline of the last run of a plan created with
 * LP_PLAN_DEBUG_TRACE.  *ctas and *cap receive the geometry: (ctas * 4 + 1)
 * rings of cap events, each event two uint64 words (globaltimer ns,
 * type << 56 | row << 24 | tile); ring (cta, role) holds counts[cta * 4 + role]
 * events (roles: 0 producer, 1 compute, 2 merge, 3 record kernel); the last
 * ring holds the prepare kernel's start and end and the record kernel's first
 * start and last end.  With events == NULL only the geometry is
 * returned.  Synchronises the plan's last stream.  LP_ESTATE without tracing. */
int lp_debug_trace(lp_plan_t plan, uint64_t* events, uint32_t* counts, int32_t* ctas, int32_t* cap);

/* Debug (tests): launches `ctas` CTAs on `stream` of device `device` that each
 * hold a whole multiprocessor's shared memory and spin for `ns` nanoseconds
 * (at most 10 s), then exit: a kernel that keeps part of the GPU busy beside
 * a run on another stream.  LP_EINVAL for a bad count or duration. */
int lp_debug_occupy(int32_t device, int32_t ctas, int64_t ns, void* stream);

/* Tiles per row for this plan (ceil(V / tile elements)). */
int lp_plan_tiles_per_row(lp_plan_t plan);

/* ---- Run without any device allocation ----
 *
 * No counterpart in the design pages.  Some callers cannot call cudaMalloc: a serving
 * process whose framework reserved the whole device for its own caching
 * allocator (a raw allocation then fails or splits its pool), code called back
 * from inside such an allocator (allocating there can deadlock on its lock),
 * and runtimes that fix their device-memory budget when they start.
 * lp_plan_create needs one cudaMalloc; lp_run_static needs none.
 *
 * lp_run_static performs exactly the operation of lp_plan_create + lp_bind +
 * lp_run with `desc` and `io` (same kernels, same outputs), but its scratch
 * (control block, work queue, per-row counters, group descriptors, per-tile
 * partial results) lives in one fixed array of LP_STATIC_SCRATCH_BYTES in the
 * library's device image.  Every GPU that loads the library holds that array
 * until the process exits.
 *
 *   desc    V, V_padded, dtype, k_max, k_alt_max, max_ids, device, timeout_ns
 *           as for a plan; max_rows / max_groups must cover io->rows /
 *           io->groups.  LP_PLAN_HOST_STAGING and LP_PLAN_DEBUG_TRACE are
 *           ignored (both would allocate).
 *   io      device buffers as for lp_bind (caller-owned, same layouts).
 *   stream  a cudaStream_t (NULL = legacy default stream).
 *
 * The scratch a run needs grows with io->rows * ceil(V / tile elements)
 * (448 bytes per row tile, plus 56 bytes per row and 16 per group);
 * a run that needs more than LP_STATIC_SCRATCH_BYTES is rejected with
 * LP_ESCRATCH before anything is enqueued.  4 MiB covers, for example, 512
 * rows of a 248,448-lane BF16 vocabulary.
 *
 * The first call on a device sets that device up (it looks up the array's
 * device address and the kernels' launch shape); make that first call before
 * any stream capture on the device.  Each call clears the array's control
 * block on `stream` before its kernels, all but its run counter, which keeps
 * counting across calls: the per-tile results and record tasks that cross
 * thread blocks during a run carry the run's number, so nothing an earlier
 * call left in the array is taken for the current call's.  All calls share the one array, so calls whose
 * work can overlap on the GPU (different streams, or different host threads)
 * race and corrupt each other: serialise them on one stream.
 *
 * Returns after enqueueing.  Errors: LP_EINVAL, LP_ESHAPE, LP_EALIGN,
 * LP_EDTYPE, LP_ECAPACITY, LP_ESCRATCH, LP_ECUDA. */
#define LP_STATIC_SCRATCH_BYTES (4u << 20)
int lp_run_static(const lp_plan_desc* desc, const lp_io* io, void* stream);

/* Message of an LP_E* code. */
const char* lp_strerror(int code);

/* The last cudaError_t seen by this library in the calling thread (0 = none). */
int lp_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* LP_EPILOGUE_H */
