// lp_internal.h -- shared between the host plan code and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace lp {

// Vocabulary tile: 8192 elements (16 KiB of BF16, 32 KiB of FP32).
constexpr int kTileElems = 8192;
constexpr int kConsumerThreads = 256;   // 8 compute warps
constexpr int kThreads = kConsumerThreads + 32;  // + 1 producer warp
constexpr int kKeysPerTile = 32;        // retained sort keys per tile
constexpr int kRecordWords = 258;
constexpr int kMaxIds = 128;
constexpr int kCandCap = 256;           // tile candidate buffer (keys)

// Pipeline stages per CTA and CTAs per SM, per element type.
template <int kElt> struct StageCfg;
template <> struct StageCfg<2> { static constexpr int kStages = 4; static constexpr int kMinBlocks = 3; };
template <> struct StageCfg<4> { static constexpr int kStages = 3; static constexpr int kMinBlocks = 2; };

// Row modes (what a read row needs).
enum : int { kModeArgmax = 0, kModeLse = 1, kModeNatural = 2 };

// Group descriptor built by the prepare kernel:
//   x = first row, y = k | mode << 8 | explicit_ids << 12 | requested << 13,
//   z = top_k (natural) or id count (explicit), w = sampled token.
struct Ctrl {
    unsigned int q_head;      // queue position whose row is being split into tiles
    unsigned int q_tail;      // queue entries reserved
    int outstanding;          // rows queued or in flight, not yet decided
    unsigned int abort;       // 1: malformed groups, the stream kernel does nothing
    unsigned int never;       // never written: the forced-timeout test hook waits on it
    unsigned int pad[11];
};

struct Params {
    // problem
    const void* logits;
    long long V, Vp;      // elements
    int rows, G, T;       // T = tiles per row
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
    int* queue;           // [max_rows] entries g << 4 | j, -1 = not yet published
    int* ticket;          // [max_rows] next tile to hand out
    int* done;            // [max_rows] tiles finished
    int4* gdesc;          // [max_groups]
    float2* part_ms;      // [max_rows * T] tile (max, exp-sum)
    unsigned long long* part_keys;  // [max_rows * T * 32] tile keys, descending
    unsigned long long timeout_ns;
    unsigned int debug_flags;
};

struct LaunchCfg {
    int grid;           // persistent CTAs
    int smem_bytes;     // dynamic shared memory of the stream kernel
};

// Enqueue prepare + stream kernels (lp_kernels.cu).
cudaError_t launch_epilogue(const Params& p, int dtype, const LaunchCfg& cfg, cudaStream_t stream);
// Occupancy-derived configuration for a dtype on the current device.
cudaError_t query_launch_cfg(int dtype, LaunchCfg* cfg);

}  // namespace lp
