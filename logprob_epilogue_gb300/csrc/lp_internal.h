// lp_internal.h -- shared between the host plan code and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace lp {

// Vocabulary tile: 32 KiB of logits (16384 BF16 or 8192 FP32 elements).
constexpr int kTileBytes = 32768;
template <int ELT>
__host__ __device__ constexpr int tile_elems() { return kTileBytes / ELT; }
inline int tile_elems_of_dtype(int dtype) { return dtype == 1 ? kTileBytes / 2 : kTileBytes / 4; }
constexpr int kConsumerThreads = 256;   // 8 compute warps
constexpr int kThreads = kConsumerThreads + 64;  // + 1 producer warp + 1 selector warp
constexpr int kKeysPerTile = 32;        // natural-alternative summary entries per tile (4 per compute warp)
constexpr int kRecordWords = 258;
constexpr int kScoreWords = 43;        // prompt-scoring record: id, lp bits, rank, 20 pairs
constexpr int kScoreAlts = 20;
constexpr int kMaxIds = 128;
constexpr int kMaxShards = 8;          // vocabulary shards of lp_run_sharded
constexpr int kShardWords = 256;       // exchange-2 words per position per shard
constexpr int kTraceRoles = 4;         // debug timeline rings per CTA: producer, compute, merge, record

// Pipeline stages per CTA and CTAs per SM, per element type: three CTAs of one
// 32 KiB stage per SM give 24 compute warps per SM and keep about 14 MB of
// copies in flight, enough for the full HBM bandwidth: more stages only
// lengthen the memory queue that every dependent read (the next row of a
// verify chain, a record's gathers) waits in.
#ifndef LP_BF16_STAGES
#define LP_BF16_STAGES 1
#endif
#ifndef LP_BF16_CTAS
#define LP_BF16_CTAS 3
#endif
#ifndef LP_F32_STAGES
#define LP_F32_STAGES 1
#endif
#ifndef LP_F32_CTAS
#define LP_F32_CTAS 3
#endif
template <int kElt> struct StageCfg;
template <> struct StageCfg<2> {
    static constexpr int kStages = LP_BF16_STAGES;
    static constexpr int kMinBlocks = LP_BF16_CTAS;
};
template <> struct StageCfg<4> {
    static constexpr int kStages = LP_F32_STAGES;
    static constexpr int kMinBlocks = LP_F32_CTAS;
};

// done[row] bit set once the row's parent has accepted (depth-0 rows: by the
// prepare kernel); the row is decided by whichever increment completes
// T + kParentDone.
constexpr int kParentDone = 1 << 24;
// tclaim[row] offset that ends read-ahead claims on the row.
constexpr unsigned kClosed = 1u << 30;

// Row modes (what a read row needs).
enum : int { kModeArgmax = 0, kModeLse = 1, kModeNatural = 2, kModeRecord = 3 };

// Run control block; each hot word sits in its own 128-byte line.
//
// Work items are (queue position, tile) pairs.  Positions [0, fresh_rows) hold
// the depth-0 rows written by the prepare kernel ("fresh" items f = pos*T +
// tile, handed out by fresh_next); rows appended after an acceptance take
// positions fresh_rows + j ("chained" items c = j*T + tile, handed out by
// chain_next, in order, before any fresh item once their row is appended).
//
// Read-ahead (plans with LP_PLAN_READ_AHEAD): a producer that streamed a
// tile of a row with a successor in its group may, while it has nothing else
// to do, stream tiles of that successor before the row is decided, claimed
// one at a time through the successor's claim counter (tclaim).
struct Ctrl {
    unsigned int fresh_next;  // fresh items handed out
    unsigned int pad0[31];
    unsigned int chain_next;  // chained items claimed (a claim may run ahead of chain_tail)
    unsigned int pad1[31];
    unsigned int chain_tail;  // chained rows reserved (their queue entries follow)
    unsigned int pad2[31];
    int outstanding;          // groups whose acceptance is not complete
    unsigned int pad3[31];
    unsigned int fresh_rows;  // depth-0 rows (set by the prepare kernel)
    unsigned int abort;       // 1: malformed groups, the stream kernel does nothing
    unsigned int never;       // never written: the forced-timeout test hook waits on it
    unsigned int chain_max;   // rows that acceptances can append at most (the read groups' drafts)
    unsigned int pad4[28];
    unsigned int rec_count;   // record tasks appended (rec_tasks[0, rec_count))
    unsigned int pad5[31];
    unsigned int rec_claim;   // record tasks claimed by producers (a claim may run ahead of rec_count)
    unsigned int pad6[31];
    unsigned int epoch;       // run number, advanced by the prepare kernel (never 0 or all ones); the
                              // tile partials and record tasks of a run carry it
    unsigned int pad7[31];
    unsigned int retired;     // stream CTAs that left their slot to the record kernel early
    unsigned int pad8[31];
};

struct Params {
    // problem
    const void* logits;
    long long V, Vp;      // elements
    int rows, G, T;       // T = tiles per row
    int elt;              // bytes per logit (2 or 4)
    int stream_grid;      // CTAs of the stream kernel
    int k_max, k_alt_max, max_ids;
    // inputs
    const int* indptr;
    const int* drafts;
    const int* sampled;
    const int* requested;
    const int* top_k;
    const int* token_ids;
    const int* id_counts;
    // outputs
    int* records;
    int* accepted;
    int* emitted;
    float* lse_out;
    unsigned int* status;
    // scratch
    Ctrl* ctrl;
    unsigned long long* queue;  // [max_rows] work queue (see queue_entry), all ones = not yet published
    unsigned int* tclaim; // [max_rows] tiles of the row claimed by read-ahead; kClosed added once
                          // the row's parent is decided
    int* done;            // [max_rows] tiles finished; with read-ahead, plus kParentDone once the row
                          // must be decided (depth-0 rows from the start, others when their parent accepts)
    unsigned long long* row_best;   // [max_rows] best (argmax) key over the finished tiles
    int4* gdesc;          // [max_groups] x = first row, y = k | mode << 8 | explicit << 12 |
                          // requested << 13, z = top_k or id count, w = sampled token
    ulonglong2* rec_tasks;  // [max_rows * 2] compact list of the records to build, appended by the
                            // deciders: words epoch << 32 | (chosen token, row, group descriptor word |
                            // count << 16, group)
    ulonglong2* part_ms;  // [max_rows * T * 8] (epoch << 32 | max bits, epoch << 32 | exp-sum bits) of
                          // each compute warp's share of a tile
    int2* part_rank;      // [max_rows * T * 8] prompt scoring: (lanes above the target's logit, the
                          // smallest such logit's bits) of each compute warp's share of a tile
    unsigned long long* part_keys;  // [max_rows * T * 32] natural tiles: each compute warp's 4 largest
                                    // thread maxima, (ord32 << 32) | (tile << 8) | thread; 0 = none
    unsigned long long timeout_ns;
    unsigned int debug_flags;
    int host_logits;      // 1: logits is pinned host memory mapped into the device's address space;
                          // tiles are copied with cp.async (16-byte copies) instead of TMA bulk copies
    int build_records;    // 1: the record kernel runs beside the stream kernel (0: the sharded kernels
                          // build the records after it)
    int read_ahead;       // 0: rows past a group's emitted prefix are never read
    // prompt scoring (targets != nullptr): group g is row g alone, k = 0, 20
    // natural alternatives, chosen token targets[g]; records go to score_records
    const int* eos;       // [G] or null: commit clipping at an emitted EOS token
    const int* budget;    // [G] or null: commit clipping at the output budget
    const int* targets;
    int* score_records;   // [rows, 43]
    int done_last;        // done[row] before the increment that completes a row: T - 1, plus
                          // kParentDone with read-ahead
    // optional timeline (nullptr unless the plan traces)
    unsigned long long* trace;    // [(trace_ctas * 3 + 1) * trace_cap * 2]
    unsigned int* trace_count;    // [trace_ctas * 3]
    int trace_cap;
    int trace_ctas;
};

// Stochastic chain verification (lp_chain.cu).
struct ChainParams {
    const void* logits;   // [rows, Vp] of the plan's dtype
    long long V, Vp;
    int rows, G, k_max;
    const int* indptr;    // [G + 1]
    const int* drafts;    // [rows]
    const float* q;       // [rows, Vp] draft laws (FP32)
    const float* temp;    // [G]
    const float* u;       // [rows] acceptance uniforms
    const float* r;       // [G] draw uniforms
    int* accepted;        // [G]
    int* emitted;         // [rows]
    float* lse_out;       // [rows] or null: lse(x / t) of the rows read
    unsigned int* status;
};

struct LaunchCfg {
    int grid;           // persistent CTAs
    int smem_bytes;     // dynamic shared memory of the stream kernel
    int sms;            // multiprocessors of the device
};

// Enqueue the prepare, stream and record kernels (lp_kernels.cu); records =
// false leaves the record kernel out (the sharded path builds the records).
cudaError_t launch_epilogue(const Params& p, int dtype, const LaunchCfg& cfg, cudaStream_t stream,
                            bool records = true);
// Enqueue the vocabulary-sharded record kernels after launch_epilogue(..., false):
// exchange 1 into x1 [rows * S], exchange 2 into x2 [rows * S * 256], the merge.
cudaError_t launch_shard_records(const Params& p, int dtype, const LaunchCfg& cfg, int S, float2* x1, int* x2,
                                 cudaStream_t stream);
// Enqueue stochastic chain verification (one 512-thread CTA per group at a time).
cudaError_t launch_chain(const ChainParams& p, int dtype, int sms, cudaStream_t stream);
// Test hook: `ctas` CTAs that each hold a multiprocessor's shared memory for `ns`.
cudaError_t launch_occupy(int ctas, unsigned long long ns, cudaStream_t stream);
// Occupancy-derived configuration for a dtype on the current device.
cudaError_t query_launch_cfg(int dtype, LaunchCfg* cfg);

}  // namespace lp
