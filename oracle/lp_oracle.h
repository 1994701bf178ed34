/*
 * lp_oracle.h -- plain CPU oracle for the generation-logprob and greedy
 * speculative-acceptance epilogue.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or constant with the
 * CUDA library: every constant below is restated here on purpose.
 *
 * What it computes (sources: "logprobs-design.md", the generation-logprob
 * contract, and "mtp-design.md", section "A speculative round is a state
 * transaction", steps 2-3):
 *
 *   - lse   = log(sum_v exp(x_v)) over the V unpadded lanes, in FP64, then
 *             rounded to FP32 (round to nearest even).
 *   - lp_v  = fl32(x_v - lse), an FP32 subtraction; a -0 result is reported
 *             as +0 (logprobs-design.md normalises the sign of a zero result).
 *   - natural alternatives: all v sorted by (lp_v descending, v ascending),
 *             the first min(K, V) reported.
 *   - explicit IDs: lp of each caller ID, in caller order.
 *   - greedy acceptance: a = number of leading drafts equal to their row's
 *             argmax over raw logits (smallest ID among equal maxima, -0 and
 *             +0 equal); the group emits rows 0..a.
 *   - record: int32[258] = chosen id, chosen lp bits, then (id, lp bits)
 *             pairs; unused pairs are (-1, 0x7FC00000).
 *   - prompt scoring (logprobs-design.md, the prompt-logprobs paragraphs):
 *             per target row, int32[43] = the actual token id, its lp bits,
 *             its rank (1 + the number of lanes whose reported lp is strictly
 *             greater), then the 20 natural alternatives as (id, lp bits)
 *             pairs.  A row whose target is -1 (or any id outside [0, V))
 *             writes id -1, NaN bits, rank 0 and alternative ids -1.
 *
 *   - stochastic chain verification (mtp-design.md, "Sampling correctness"):
 *             see orc_chain_verify.
 *
 * Logits are passed as FP32 (BF16 inputs are widened exactly by the caller).
 * -Inf lanes (a masked vocabulary) are allowed where a row keeps a finite lane;
 * the oracle is not defined for NaN or +Inf.
 */
#ifndef LP_ORACLE_H
#define LP_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Record geometry: chosen pair + 128 alternative pairs = 258 int32 words. */
#define ORC_RECORD_WORDS 258
#define ORC_MAX_PAIRS 128
#define ORC_NAN_BITS 0x7FC00000u

/* Status bits (same meaning as the library's device status word). */
#define ORC_STATUS_BAD_ID 0x1u
#define ORC_STATUS_BAD_TOKEN 0x2u
#define ORC_STATUS_BAD_COUNT 0x4u
#define ORC_STATUS_BAD_GROUP 0x8u

/* log-sum-exp of x[0..V) computed in double, rounded to float. V >= 1. */
float orc_lse(const float* x, int64_t V);

/* Index of the largest x (smallest index among equal maxima). V >= 1. */
int32_t orc_argmax(const float* x, int64_t V);

/* fl32(x - lse) with -0 reported as +0. */
float orc_logprob(float x, float lse);

/*
 * Natural alternatives: sorts all V lanes by (fl32(x - lse) desc, id asc)
 * with a full stable sort and writes the first n = min(K, V) ids and
 * logprobs.  Returns n.
 */
int32_t orc_topk(const float* x, int64_t V, float lse, int32_t K, int32_t* ids, float* lps);

/* Whole epilogue over one logit block (all pointers are host memory). */
typedef struct {
    const float* logits;          /* [rows, Vp]; lanes >= V are ignored */
    int64_t rows, V, Vp;
    int32_t groups;
    const int32_t* group_indptr;   /* [groups+1] */
    const int32_t* draft_tokens;   /* [rows] */
    const int32_t* sampled_tokens; /* [groups]; <0 -> argmax */
    const int32_t* requested;      /* [groups]; nonzero = report */
    const int32_t* top_k;          /* [groups] */
    const int32_t* token_ids;      /* [groups, 128] */
    const int32_t* id_counts;      /* [groups]; 0 -> natural */
    int32_t k_max;                 /* largest allowed drafts per group */
    int32_t k_alt_max;             /* largest allowed K (natural alternatives) */
    int32_t max_ids;               /* largest allowed explicit-ID count */
    int32_t* records;              /* [rows, 258]; only emitted flagged rows written */
    int32_t* accepted;             /* [groups] */
    int32_t* emitted_tokens;       /* [rows]; -1 for rows not emitted */
    float* lse_out;                /* [rows] or NULL; written for rows whose lse is computed */
    uint32_t* status;              /* out: status bits */
    int64_t* rows_read;            /* out (optional): logit rows the path had to read */
    /* Commit clipping ("mtp-design.md", a speculative round, step 4 and the
     * paragraph after it), both optional (NULL = none): */
    const int32_t* eos_tokens;     /* [groups]; the emitted prefix ends at this token (< 0 = none) */
    const int32_t* budgets;        /* [groups]; at most this many tokens emitted; <= 0 = at the limit */
} orc_io;

/* Runs the epilogue; groups are split over `threads` host threads (<=1: one).
 * Returns 0, or -1 on a NULL required pointer. */
int orc_epilogue(const orc_io* io, int threads);

/* Prompt scoring record geometry: id, lp bits, rank, 20 (id, lp bits) pairs. */
#define ORC_SCORE_WORDS 43
#define ORC_SCORE_ALTS 20

/* 1 + number of lanes v in [0, V) with fl32(x_v - lse) > lp. */
int32_t orc_rank(const float* x, int64_t V, float lse, float lp);

/* Prompt scoring of rows [0, rows): records [rows, 43]; lse_out [rows] or NULL
 * (written for valid rows); status gets ORC_STATUS_BAD_TOKEN for a target >= V.
 * Returns 0, or -1 on a NULL required pointer. */
int orc_score(const float* logits, int64_t rows, int64_t V, int64_t Vp, const int32_t* targets,
              int32_t* records, float* lse_out, uint32_t* status, int threads);

/* Stochastic chain verification ("mtp-design.md", "Sampling correctness":
 * accept each draft with probability min(1, p/q); on the first rejection draw
 * from the normalised positive residual max(p - q, 0); after full acceptance
 * draw the bonus token from the target law).  Groups as in orc_io: group g
 * holds k drafts on rows r0..r0+k-1 and its bonus row r0+k.  For row j:
 *   p_j(v) = exp(x_j(v)/t - lse(x_j/t)) over the V lanes, t = temperature[g]
 *            (FP64 throughout);
 *   q_j    = draft_probs row r0+j: the law that drew draft d_j (j < k);
 *   draft j is accepted iff u[r0+j] * q_j(d_j) < p_j(d_j), i.e. u < p/q;
 *   a      = the number of leading accepted drafts;
 *   the last token is drawn with r[g] in [0, 1) by inverse CDF over ids in
 *   ascending order: the smallest v whose running sum of weights exceeds
 *   r[g] * (total weight), the weights being max(p_a - q_a, 0) when a < k
 *   (p_a itself if that residual has no mass) and p_k when a == k.
 * Outputs: accepted[g] = a; emitted[r0+j] = d_j for j < a, the drawn token at
 * j = a, -1 after.  The random numbers are inputs.  Returns 0, or -1 on a NULL
 * pointer or a temperature that is not > 0. */
int orc_chain_verify(const float* logits, int64_t rows, int64_t V, int64_t Vp, int32_t groups,
                     const int32_t* group_indptr, const int32_t* draft_tokens, const float* draft_probs,
                     const float* temperature, const float* u, const float* r, int32_t* accepted,
                     int32_t* emitted);

#ifdef __cplusplus
}
#endif

#endif
