// lp_kernels.cu -- sm_103a kernels of the logprob / greedy-acceptance epilogue.
//
// Two launches per run, both on the caller's stream:
//
//  lp_prepare_kernel (1 CTA)
//    validates group_indptr, resolves each group's request (natural
//    alternatives, explicit ids or argmax only), finishes groups that need no
//    logits, resets the per-row counters and writes the depth-0 work queue:
//    row 0 of every group that must be read.
//
//  lp_stream_kernel (persistent, PDL-overlapped with the prepare kernel),
//  warp-specialised CTAs of 10 warps:
//    - producer warp: draws work items (queue position, tile) from one global
//      counter and streams each 8192-element vocabulary tile into a
//      shared-memory stage with a TMA bulk copy (cp.async.bulk, mbarrier
//      completion, L2 evict-first);
//    - 8 compute warps: reduce a tile to its FP32 max, exp-sum (ex2) relative
//      to that max, argmax key and, for rows that report natural alternatives,
//      the tile's best 32 packed sort keys
//          key = ord32(x) << 32 | (0xFFFFFFFF - id),
//      ord32 being the monotone float -> uint map with -0 folded into +0;
//      results go to a shared-memory ring;
//    - merge warp: publishes tile results to global memory, counts the row's
//      finished tiles and, on the last one, merges the row: argmax -> greedy
//      acceptance (on acceptance the next row of the group is appended to the
//      queue, so rows past the accepted prefix are never read), then
//      lse = M + log(sum s_t exp(m_t - M)), the chosen token's logprob, the
//      top-K natural alternatives or the explicit-id gather, and the 258-word
//      record.
//
// Sources: "logprobs-design.md" (generation-logprob contract; the four-launch
// reduction paragraph: FP32 tile maxima and exponential sums, a per-position
// normalisation, tiles keeping their best 32 integer sort keys over reported
// FP32 logprobs and inverse ids, ties from the subtraction included, equal
// values at the cutoff taking the smallest ids, signed zero normalised, padded
// lanes excluded, explicit ids gathered from raw logits) and "mtp-design.md"
// ("A speculative round is a state transaction", steps 2-3).
//
// Exactness of the natural alternatives with per-tile top-32 by RAW key:
// fl32(x - lse) is non-decreasing in x, so the global raw top-32 holds every
// lane whose logprob exceeds the K-th value L; lanes with logprob == L may sit
// below it (ties created by the subtraction).  If the 32nd raw key's logprob
// is below L, every lane with logprob >= L is inside the raw top-32 and a sort
// of those 32 by (logprob, inverse id) is exact.  Otherwise the lanes equal to
// L are collected tile by tile in id order; a tile can hide such a lane only
// if its own 32nd key has logprob == L, and only such tiles are re-read.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "lp_internal.h"

namespace lp {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNegInf = -__builtin_huge_valf();
constexpr unsigned kStatusBadId = 0x1u, kStatusBadToken = 0x2u, kStatusBadCount = 0x4u,
                   kStatusBadGroup = 0x8u, kStatusTimeout = 0x10u;
constexpr unsigned kDebugForceTimeout = 0x100u;
constexpr unsigned kUnusedBits = 0x7FC00000u;

// ------------------------------------------------------------------ helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Monotone map float -> uint32 (x already free of -0).
__device__ __forceinline__ uint32_t ord32(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float unord32(uint32_t o) {
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

__device__ __forceinline__ unsigned long long make_key(float x, uint32_t id) {
    x = __fadd_rn(x, 0.0f);  // -0 -> +0
    return (static_cast<unsigned long long>(ord32(x)) << 32) | static_cast<unsigned long long>(~id);
}

__device__ __forceinline__ float key_value(unsigned long long k) { return unord32(static_cast<uint32_t>(k >> 32)); }
__device__ __forceinline__ uint32_t key_id(unsigned long long k) { return ~static_cast<uint32_t>(k); }

// Reported logprob: fl32(x - lse), -0 -> +0.
__device__ __forceinline__ float logprob(float x, float lse) { return __fadd_rn(__fsub_rn(x, lse), 0.0f); }

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void cbar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Barrier over the compute threads that also ORs a predicate across them.
__device__ __forceinline__ bool cbar_or(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, 1, 256, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

template <typename T>
__device__ __forceinline__ T vload(const T* p) { return *reinterpret_cast<const volatile T*>(p); }
template <typename T>
__device__ __forceinline__ void vstore(T* p, T v) { *reinterpret_cast<volatile T*>(p) = v; }

// ---- optional device timeline (plans created with the trace flag)
//
// Each CTA has three event rings (producer, compute, merge warp) of
// p.trace_cap events; an event is (globaltimer ns, type << 56 | row << 24 | tile).
enum : unsigned { kTrKernel = 1, kTrClaim, kTrIssue, kTrTileStart, kTrTileEnd, kTrPublish, kTrMergeStart,
                  kTrDecision, kTrMergeEnd, kTrPrepStart, kTrPrepEnd, kTrExit, kTrTileB1, kTrTileB2 };

__shared__ unsigned g_trace_n[3];  // per-CTA event counts (producer, compute, merge)

__device__ __forceinline__ void trace(const Params& p, unsigned type, int row, int tile, bool writer) {
    if (p.trace == nullptr || !writer) return;
    const int role = type == kTrClaim || type == kTrIssue || type == kTrExit ? 0
                   : (type == kTrTileStart || type == kTrTileEnd || type == kTrKernel || type == kTrTileB1 ||
                      type == kTrTileB2) ? 1 : 2;
    unsigned* cnt = g_trace_n + role;
    const unsigned i = *cnt;
    if (i >= (unsigned)p.trace_cap) return;
    *cnt = i + 1;
    p.trace_count[blockIdx.x * 3 + role] = i + 1;
    unsigned long long* e = p.trace + (((size_t)blockIdx.x * 3 + role) * p.trace_cap + i) * 2;
    e[0] = globaltimer();
    e[1] = ((unsigned long long)type << 56) | ((unsigned long long)(row & 0xFFFFFFFF) << 24) |
           (unsigned long long)(tile & 0xFFFFFF);
}

// ---- mbarrier / bulk copy (PTX ISA: mbarrier, cp.async.bulk)

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking probe of the phase of `parity`.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase of `parity`; false if the deadline passed first.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned long long deadline) {
    for (uint32_t i = 0;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 63u && globaltimer() > deadline) return false;
    }
}

__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar,
                                          uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// ---- warp / block reductions (block = the 256 compute threads)

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}
__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long w = __shfl_xor_sync(kFull, v, o);
        v = w > v ? w : v;
    }
    return v;
}

// Sorts one value per lane in descending order across the warp (bitonic).
template <typename T>
__device__ __forceinline__ T warp_sort_desc(T v, int lane) {
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const T p = __shfl_xor_sync(kFull, v, j);
            const bool desc_block = (lane & k) == 0;
            const bool lower = (lane & j) == 0;
            const bool take_max = desc_block == lower;
            v = take_max ? (p > v ? p : v) : (p < v ? p : v);
        }
    }
    return v;
}

// Sorts a bitonic sequence (one value per lane) in descending order.
__device__ __forceinline__ unsigned long long warp_bitonic_clean_desc(unsigned long long v, int lane) {
#pragma unroll
    for (int j = 16; j > 0; j >>= 1) {
        const unsigned long long p = __shfl_xor_sync(kFull, v, j);
        const bool lower = (lane & j) == 0;
        v = lower ? (p > v ? p : v) : (p < v ? p : v);
    }
    return v;
}

constexpr int kTasks = 64;  // record tasks a CTA can hold for its compute warps
constexpr int kMaxStages = 8;
static_assert(StageCfg<2>::kStages <= kMaxStages && StageCfg<4>::kStages <= kMaxStages, "stage count");

// One tile result handed from the compute warps to the merge warp.
struct ResultSlot {
    int4 info;                       // row, tile, queue entry (< 0: no more tiles), mode
    float M, S;                      // tile max and sum exp(x - M)
    unsigned long long keys[kKeysPerTile];  // descending; keys[0] = tile argmax key
};

struct Shared {
    uint64_t full[kMaxStages];       // stage filled (producer + TMA)
    uint64_t empty[kMaxStages];      // stage released (8 compute warps)
    uint64_t rfull[kRing];           // result written (8 compute warps)
    uint64_t rempty[kRing];          // result consumed (merge warp)
    int4 info[kMaxStages];           // work item of each stage
    ResultSlot res[kRing];
    union {
        unsigned long long cand[kCandCap];  // natural-alternative candidates of a tile
        unsigned long long lists[8][32];    // per-warp partial top-32 lists of a record task
    };
    unsigned long long wkey[2][8];   // per-warp partials, double-buffered by tile parity
    float wM[2][8];
    float wS[2][8];
    float wTheta[2][8];
    int ncand[2];
    int wcnt[2][8];                  // candidates per warp, double-buffered by tile parity
    unsigned long long red_u64[8];
    double red_d[8];
    float red_f[8];
    float red_f2[8];
    int red_i[8];
    float lse;
    float xchosen;
    int rec[kRecordWords + 2];       // record being assembled by the compute warps
    int2 batch[kRing];               // (row, queue entry) of the tiles in a merge-warp batch
    int mrec[kRecordWords + 2];      // record assembled by the merge warp (task ring full)
    int4 task[kTasks];               // record tasks: (row, chosen, queue entry, kModeRecord)
    unsigned task_head;              // tasks taken by the compute warps
    unsigned task_tail;              // tasks pushed by the merge warp
    unsigned task_snap[2];           // task_tail seen at a tile's first barrier (by tile parity)
};

// ---- block reductions over the 256 compute threads (slow path only)

__device__ __forceinline__ float block_max_f(float v, Shared& sm, int lane, int warp) {
    v = warp_max_f(v);
    if (lane == 0) sm.red_f[warp] = v;
    cbar();
    float r = sm.red_f[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) r = fmaxf(r, sm.red_f[i]);
    cbar();
    return r;
}

__device__ __forceinline__ int block_sum_i(int v, Shared& sm, int lane, int warp) {
    v = warp_sum_i(v);
    if (lane == 0) sm.red_i[warp] = v;
    cbar();
    int r = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) r += sm.red_i[i];
    cbar();
    return r;
}

__device__ __forceinline__ double block_sum_d(double v, Shared& sm, int lane, int warp) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    if (lane == 0) sm.red_d[warp] = v;
    cbar();
    double r = 0.0;
#pragma unroll
    for (int i = 0; i < 8; ++i) r += sm.red_d[i];
    cbar();
    return r;
}

// Exclusive prefix sum over the 256 compute threads; *total = the sum.
__device__ __forceinline__ int block_excl_scan_i(int v, int* total, Shared& sm, int lane, int warp) {
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) sm.red_i[warp] = incl;
    cbar();
    int before = 0, all = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int t = sm.red_i[i];
        before += (i < warp) ? t : 0;
        all += t;
    }
    cbar();
    *total = all;
    return before + incl - v;
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

// ---- tile element access
//
// Full tiles: thread i owns the 16-byte vectors c*256 + i (c = 0..NCH-1), so
// element k = c*EPV + s of the thread is tile element (c*256 + i)*EPV + s.
// Partial tiles (the last tile of a row): element k of thread i is tile element
// k*256 + i, masked beyond the valid count.  Both orders are ascending in k.

template <int ELT>
struct TileLayout {
    static constexpr int EPV = 16 / ELT;          // elements per 16-byte vector
    static constexpr int NCH = kTileBytes / 16 / kConsumerThreads;  // vectors per thread (8)
    static constexpr int EPT = EPV * NCH;         // elements per thread (64 BF16, 32 FP32)
};

template <int ELT>
__device__ __forceinline__ int tile_elem_id(bool full, int k, int tid) {
    using L = TileLayout<ELT>;
    return full ? ((k / L::EPV) * kConsumerThreads + tid) * L::EPV + (k % L::EPV) : k * kConsumerThreads + tid;
}

// 16-byte shared-memory load through an explicit shared-space address.
__device__ __forceinline__ uint4 lds128(const void* p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_u32(p)));
    return v;
}

__device__ __forceinline__ int atomic_add_shared(int* p, int v) {
    int old;
    asm volatile("atom.shared.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(smem_u32(p)), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void st_shared_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.shared.u64 [%0], %1;" ::"r"(smem_u32(p)), "l"(v) : "memory");
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Register copy of a thread's tile elements: FP32 as floats, BF16 kept packed
// two per word (element k in the low half of word k/2 when k is even).
template <int ELT>
struct TileRegs;

template <>
struct TileRegs<4> {
    static constexpr int kN = TileLayout<4>::EPT;
    float x[kN];
    __device__ __forceinline__ float get(int k) const { return x[k]; }
    __device__ __forceinline__ float max() const {
        float m = x[0];
#pragma unroll
        for (int k = 1; k < kN; ++k) m = fmaxf(m, x[k]);
        return m;
    }
    __device__ __forceinline__ void load(const unsigned char* stage, bool full, int nv, int tid) {
        if (full) {
#pragma unroll
            for (int c = 0; c < TileLayout<4>::NCH; ++c) {
                const uint4 v = lds128(stage + (size_t)(c * kConsumerThreads + tid) * 16);
                x[c * 4 + 0] = __uint_as_float(v.x);
                x[c * 4 + 1] = __uint_as_float(v.y);
                x[c * 4 + 2] = __uint_as_float(v.z);
                x[c * 4 + 3] = __uint_as_float(v.w);
            }
        } else {
            const float* f = reinterpret_cast<const float*>(stage);
#pragma unroll
            for (int k = 0; k < kN; ++k) {
                const int e = k * kConsumerThreads + tid;
                x[k] = e < nv ? f[e] : kNegInf;
            }
        }
    }
};

__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

template <>
struct TileRegs<2> {
    static constexpr int kN = TileLayout<2>::EPT;
    uint32_t w[kN / 2];
    __device__ __forceinline__ float get(int k) const { return (k & 1) ? bf16_hi(w[k >> 1]) : bf16_lo(w[k >> 1]); }
    __device__ __forceinline__ float max() const {
        uint32_t m = w[0];
#pragma unroll
        for (int i = 1; i < kN / 2; ++i) m = bf16x2_max(m, w[i]);
        return fmaxf(bf16_lo(m), bf16_hi(m));
    }
    __device__ __forceinline__ void load(const unsigned char* stage, bool full, int nv, int tid) {
        if (full) {
#pragma unroll
            for (int c = 0; c < TileLayout<2>::NCH; ++c) {
                const uint4 v = lds128(stage + (size_t)(c * kConsumerThreads + tid) * 16);
                w[c * 4 + 0] = v.x;
                w[c * 4 + 1] = v.y;
                w[c * 4 + 2] = v.z;
                w[c * 4 + 3] = v.w;
            }
        } else {
            const unsigned short* h = reinterpret_cast<const unsigned short*>(stage);
#pragma unroll
            for (int i = 0; i < kN / 2; ++i) {
                const int e0 = (2 * i) * kConsumerThreads + tid, e1 = (2 * i + 1) * kConsumerThreads + tid;
                const uint32_t lo = e0 < nv ? h[e0] : 0xFF80u;  // -inf in masked lanes
                const uint32_t hi = e1 < nv ? h[e1] : 0xFF80u;
                w[i] = lo | (hi << 16);
            }
        }
    }
};

// Streaming passes over a full stage (thread i reads vectors c*256 + i).
template <int ELT>
__device__ __forceinline__ float stage_max(const unsigned char* sp, int tid) {
    constexpr int NCH = TileLayout<ELT>::NCH;
    if constexpr (ELT == 2) {
        uint32_t a = 0xFF80FF80u, b = 0xFF80FF80u;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const uint4 v = lds128(sp + (size_t)(c * kConsumerThreads + tid) * 16);
            a = bf16x2_max(a, bf16x2_max(v.x, v.y));
            b = bf16x2_max(b, bf16x2_max(v.z, v.w));
        }
        a = bf16x2_max(a, b);
        return fmaxf(bf16_lo(a), bf16_hi(a));
    } else {
        float a = kNegInf, b = kNegInf;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const uint4 v = lds128(sp + (size_t)(c * kConsumerThreads + tid) * 16);
            a = fmaxf(a, fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)));
            b = fmaxf(b, fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
        }
        return fmaxf(a, b);
    }
}

template <int ELT>
__device__ __forceinline__ float stage_expsum(const unsigned char* sp, int tid, float mb) {
    constexpr int NCH = TileLayout<ELT>::NCH;
    float s0 = 0.0f, s1 = 0.0f, s2 = 0.0f, s3 = 0.0f;
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
        const uint4 v = lds128(sp + (size_t)(c * kConsumerThreads + tid) * 16);
        if constexpr (ELT == 2) {
            s0 += ex2(fmaf(bf16_lo(v.x), kLog2e, -mb)) + ex2(fmaf(bf16_hi(v.x), kLog2e, -mb));
            s1 += ex2(fmaf(bf16_lo(v.y), kLog2e, -mb)) + ex2(fmaf(bf16_hi(v.y), kLog2e, -mb));
            s2 += ex2(fmaf(bf16_lo(v.z), kLog2e, -mb)) + ex2(fmaf(bf16_hi(v.z), kLog2e, -mb));
            s3 += ex2(fmaf(bf16_lo(v.w), kLog2e, -mb)) + ex2(fmaf(bf16_hi(v.w), kLog2e, -mb));
        } else {
            s0 += ex2(fmaf(__uint_as_float(v.x), kLog2e, -mb));
            s1 += ex2(fmaf(__uint_as_float(v.y), kLog2e, -mb));
            s2 += ex2(fmaf(__uint_as_float(v.z), kLog2e, -mb));
            s3 += ex2(fmaf(__uint_as_float(v.w), kLog2e, -mb));
        }
    }
    return (s0 + s1) + (s2 + s3);
}

template <int ELT>
__device__ __forceinline__ float partial_max(const unsigned char* sp, int nv, int tid) {
    TileRegs<ELT> x;
    x.load(sp, false, nv, tid);
    return x.max();
}

template <int ELT>
__device__ __forceinline__ float partial_expsum(const unsigned char* sp, int nv, int tid, float mb) {
    TileRegs<ELT> x;
    x.load(sp, false, nv, tid);
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < TileRegs<ELT>::kN; ++k) s += ex2(fmaf(x.get(k), kLog2e, -mb));
    return s;
}

template <int ELT>
__device__ __forceinline__ float load_logit(const Params& p, int row, long long id) {
    const long long off = (long long)row * p.Vp + id;
    if constexpr (ELT == 4) {
        return __ldg(reinterpret_cast<const float*>(p.logits) + off);
    } else {
        const unsigned short b = __ldg(reinterpret_cast<const unsigned short*>(p.logits) + off);
        return __uint_as_float(static_cast<uint32_t>(b) << 16);
    }
}

// Work-queue entry: high word = g << 4 | j (group, row within the group),
// low word = row | mode << 28.  All ones = reserved but not yet published.
__device__ __forceinline__ unsigned long long queue_entry(int gj, int row, int mode) {
    return ((unsigned long long)(uint32_t)gj << 32) | (unsigned long long)(uint32_t)(row | (mode << 28));
}

// ------------------------------------------------------------------ prepare

__global__ void __launch_bounds__(1024) lp_prepare_kernel(Params p) {
    asm volatile("griddepcontrol.launch_dependents;");
    if (p.trace != nullptr && threadIdx.x == 0) {
        unsigned long long* e = p.trace + ((size_t)p.trace_ctas * 3) * p.trace_cap * 2;
        e[0] = globaltimer();
        e[1] = (unsigned long long)kTrPrepStart << 56;
    }
    __shared__ int s_warp[32];
    __shared__ int s_total;
    __shared__ int s_base;
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    for (int r = tid; r < p.rows; r += blockDim.x) {
        p.done[r] = 0;
        p.queue[r] = ~0ull;
        p.row_best[r] = 0ull;
    }
    if (tid == 0) *p.status = 0u;
    const int G = p.G;
    int ok = 1;
    if (G > 0) {
        if (tid == 0) ok = (p.indptr[0] >= 0) && (p.indptr[G] <= p.rows);
        for (int g = tid; g < G; g += blockDim.x) {
            const int size = p.indptr[g + 1] - p.indptr[g];
            if (size < 1 || size - 1 > p.k_max) ok = 0;
        }
    }
    ok = __syncthreads_and(ok);
    if (!ok) {
        if (tid == 0) {
            atomicOr(p.status, kStatusBadGroup);
            p.ctrl->abort = 1u;
            p.ctrl->next_item = 0u;
            p.ctrl->q_tail = 0u;
            p.ctrl->outstanding = 0;
        }
        return;
    }
    if (tid == 0) s_base = 0;
    __syncthreads();
    unsigned st = 0;
    for (int g0 = 0; g0 < G; g0 += blockDim.x) {
        const int g = g0 + tid;
        int need = 0, row0 = 0, mode0 = 0;
        if (g < G) {
            const int r0 = p.indptr[g];
            const int k = p.indptr[g + 1] - r0 - 1;
            const int req = p.requested[g] != 0;
            const int samp = p.sampled[g];
            int cnt = p.id_counts[g];
            int K = p.top_k[g];
            int mode = kModeArgmax, kc = 0, ids = 0;
            if (req) {
                if (cnt < 0 || cnt > p.max_ids) {
                    st |= kStatusBadCount;
                    cnt = cnt < 0 ? 0 : p.max_ids;
                }
                if (cnt > 0) {
                    ids = 1;
                    kc = cnt;
                    mode = kModeLse;
                } else {
                    if (K < 0 || K > p.k_alt_max) {
                        st |= kStatusBadCount;
                        K = K < 0 ? 0 : p.k_alt_max;
                    }
                    kc = K;
                    mode = K > 0 ? kModeNatural : kModeLse;
                }
            }
            need = req || k >= 1 || samp < 0;
            if (!need) {
                if (samp >= p.V) st |= kStatusBadToken;
                p.emitted[r0] = samp;
                p.accepted[g] = 0;
            }
            p.gdesc[g] = make_int4(r0, k | (mode << 8) | (ids << 12) | (req << 13), kc, samp);
            row0 = r0;
            mode0 = mode;
        }
        const unsigned bal = __ballot_sync(kFull, need);
        const int pos_in_warp = __popc(bal & ((1u << lane) - 1u));
        if (lane == 0) s_warp[warp] = __popc(bal);
        __syncthreads();
        if (warp == 0) {
            const int v = (lane < (int)(blockDim.x >> 5)) ? s_warp[lane] : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(kFull, incl, o);
                if (lane >= o) incl += n;
            }
            s_warp[lane] = incl - v;
            if (lane == 31) s_total = incl;
        }
        __syncthreads();
        if (need) p.queue[s_base + s_warp[warp] + pos_in_warp] = queue_entry(g << 4, row0, mode0);
        __syncthreads();
        if (tid == 0) s_base += s_total;
        __syncthreads();
    }
    if (st) atomicOr(p.status, st);
    if (p.trace != nullptr) {
        for (int i = tid; i < p.trace_ctas * 3; i += blockDim.x) p.trace_count[i] = 0u;
    }
    if (tid == 0) {
        if (p.trace != nullptr) {
            unsigned long long* e = p.trace + ((size_t)p.trace_ctas * 3) * p.trace_cap * 2;
            e[2] = globaltimer();
            e[3] = (unsigned long long)kTrPrepEnd << 56;
        }
        p.ctrl->next_item = 0u;
        p.ctrl->q_tail = static_cast<unsigned>(s_base);
        p.ctrl->outstanding = s_base;
        p.ctrl->abort = 0u;
    }
}

// ------------------------------------------------------------------ producer
//
// Work items are numbered in queue order: item i is tile (i % T) of the row
// at queue position i / T.  Positions below q_tail exist (depth-0 rows from
// the prepare kernel, then rows appended by merges); a producer that draws an
// item of a position not yet appended waits until it is, or until no row is
// outstanding (then the run is complete).

// Items drawn per atomic: 4 while the queue holds plenty of work for every
// CTA, else 1 (short queues are latency-bound: spread a row's tiles wide).
__device__ __forceinline__ unsigned claim_size(unsigned tail_items, unsigned next) {
    return tail_items > next + 16u * gridDim.x ? 4u : 1u;
}

template <int ELT>
__device__ __noinline__ void producer_loop(const Params& p, Shared& sm, unsigned char* stages, unsigned long long t0) {
    constexpr int S = StageCfg<ELT>::kStages;
    constexpr int TILE_BYTES = kTileBytes;
    constexpr int kTE = tile_elems<ELT>();
    const unsigned long long deadline = t0 + p.timeout_ns;
    const uint64_t policy = evict_first_policy();
    Ctrl* ctrl = p.ctrl;
    const unsigned T = (unsigned)p.T;
    int stage = 0;
    uint32_t phase = 0;
    unsigned cached_tail = vload(&ctrl->q_tail);
    unsigned last_pos = 0xFFFFFFFFu;
    int cur_entry = -1, cur_row = 0, cur_mode = 0;
    // claims: the current chunk, plus (while the queue is long) the next chunk
    // with its atomic already in flight
    unsigned cur = 0, cur_n = 0, nxt = 0, nxt_n = 0;
    unsigned pre_pos = 0xFFFFFFFFu;   // queue position whose entry was prefetched
    unsigned long long pre_val = ~0ull;
    int prev_stage = -1;              // stage of the last fill and the phase bit of that fill
    uint32_t prev_phase = 0;
    for (;;) {
        int4 item = make_int4(0, 0, -1, 0);
        if (p.debug_flags & kDebugForceTimeout) {
            // Test hook: wait on a flag that nothing sets, until the limit.
            while (vload(&ctrl->never) == 0u) {
                if (globaltimer() > deadline) break;
                __nanosleep(1000);
            }
            atomicOr(p.status, kStatusTimeout);
        } else {
            if (cur_n == 0) {
                const unsigned tail_items = cached_tail * T;
                const unsigned seen = nxt_n > 0 ? nxt : cur;
                if (prev_stage >= 0 && tail_items < seen + 2u * gridDim.x) {
                    // short queue: take a tile only once the compute warps hold the
                    // previous one, so a row's tiles spread over many CTAs
                    if (!mbar_wait(&sm.empty[prev_stage], prev_phase, deadline)) {
                        atomicOr(p.status, kStatusTimeout);
                        return;
                    }
                }
                if (nxt_n > 0) {
                    cur = nxt;
                    cur_n = nxt_n;
                    nxt_n = 0;
                } else {
                    cur_n = claim_size(tail_items, seen);
                    cur = atomicAdd(&ctrl->next_item, cur_n);
                }
                if (cached_tail * T > cur + cur_n + 4u * gridDim.x) {
                    nxt_n = claim_size(cached_tail * T, cur + cur_n);
                    nxt = atomicAdd(&ctrl->next_item, nxt_n);
                }
            }
            const unsigned pos = cur / T;
            const unsigned tile = cur - pos * T;
            trace(p, kTrClaim, (int)pos, (int)tile, true);
            bool avail = pos < cached_tail;
            while (!avail) {
                cached_tail = vload(&ctrl->q_tail);
                if (pos < cached_tail) {
                    avail = true;
                    break;
                }
                if (vload(&ctrl->outstanding) <= 0) {
                    __threadfence();
                    cached_tail = vload(&ctrl->q_tail);  // final once nothing is outstanding
                    avail = pos < cached_tail;
                    break;
                }
                if (globaltimer() > deadline) {
                    atomicOr(p.status, kStatusTimeout);
                    break;
                }
                __nanosleep(20);
            }
            if (avail) {
                if (pos != last_pos) {
                    unsigned long long e = (pos == pre_pos) ? pre_val : vload(&p.queue[pos]);
                    for (uint32_t k = 0; (long long)e < 0; ++k) {  // reserved, not yet published
                        if ((k & 63u) == 63u && globaltimer() > deadline) break;
                        e = vload(&p.queue[pos]);
                    }
                    if ((long long)e < 0) {
                        atomicOr(p.status, kStatusTimeout);
                        avail = false;
                    } else {
                        cur_entry = (int)(e >> 32);
                        cur_row = (int)(e & 0x0FFFFFFFu);
                        cur_mode = (int)((e >> 28) & 3u);
                        last_pos = pos;
                    }
                }
                if (avail) {
                    item = make_int4(cur_row, (int)tile, cur_entry, cur_mode);
                    ++cur;
                    --cur_n;
                }
            }
        }
        if (!mbar_wait(&sm.empty[stage], phase ^ 1u, deadline)) {
            atomicOr(p.status, kStatusTimeout);
            return;
        }
        sm.info[stage] = item;
        if (item.z < 0) {
            mbar_arrive(&sm.full[stage]);
            trace(p, kTrExit, 0, 0, true);
            return;
        }
        const long long tbase = (long long)item.y * kTE;
        const long long rem = p.V - tbase;
        const int nv = rem < kTE ? (int)rem : kTE;
        const uint32_t bytes = (static_cast<uint32_t>(nv * ELT) + 15u) & ~15u;
        const unsigned char* src =
            reinterpret_cast<const unsigned char*>(p.logits) + ((long long)item.x * p.Vp + tbase) * ELT;
        mbar_arrive_expect_tx(&sm.full[stage], bytes);
        bulk_load(stages + (size_t)stage * TILE_BYTES, src, bytes, &sm.full[stage], policy);
        trace(p, kTrIssue, item.x, item.y, true);
        prev_stage = stage;
        prev_phase = phase;
        if (++stage == S) {
            stage = 0;
            phase ^= 1u;
        }
        // prefetch the queue entry of the next item (its load overlaps the next stage wait)
        const unsigned nidx = cur_n > 0 ? cur : (nxt_n > 0 ? nxt : 0xFFFFFFFFu);
        const unsigned npos = nidx / T;
        if (nidx != 0xFFFFFFFFu && npos != last_pos && npos != pre_pos && npos < cached_tail) {
            pre_pos = npos;
            pre_val = vload(&p.queue[npos]);
        }
    }
}

// ------------------------------------------------------------------ tile: exact slow top-32

// Element k of the calling thread (tile layout), read from the stage; -inf past nv.
template <int ELT>
__device__ __forceinline__ float stage_elem(const unsigned char* sp, bool full, int nv, int k, int tid) {
    const int e = tile_elem_id<ELT>(full, k, tid);
    if (e >= nv) return kNegInf;
    if constexpr (ELT == 4) {
        return reinterpret_cast<const float*>(sp)[e];
    } else {
        return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const unsigned short*>(sp)[e]) << 16);
    }
}

// Exact top-32 keys of a tile when a warp overflowed its candidate region
// (massive ties): the 32nd largest value v is found by walking distinct values
// down from the maximum; the result is every lane above v plus the smallest ids
// equal to v.  Reads the stage element by element (no register copy).
template <int ELT>
__device__ __forceinline__ void tile_top32_slow(const unsigned char* stage, bool full, int nv, long long tbase,
                                                Shared& sm, unsigned long long* out) {
    using L = TileLayout<ELT>;
    constexpr int N = L::EPT;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float v = __builtin_huge_valf();
    int cnt_ge = 0;
    for (int it = 0; it < 33; ++it) {
        float loc = kNegInf;
#pragma unroll 8
        for (int k = 0; k < N; ++k) {
            const float x = stage_elem<ELT>(stage, full, nv, k, tid);
            loc = (x < v && x > loc) ? x : loc;
        }
        const float vn = block_max_f(loc, sm, lane, warp);
        if (!(vn > kNegInf)) break;  // no value left below v
        v = vn;
        int c = 0;
#pragma unroll 8
        for (int k = 0; k < N; ++k) {
            const float x = stage_elem<ELT>(stage, full, nv, k, tid);
            c += (x >= v && x > kNegInf) ? 1 : 0;
        }
        cnt_ge = block_sum_i(c, sm, lane, warp);
        if (cnt_ge >= 32) break;
    }
    int c = 0;
#pragma unroll 8
    for (int k = 0; k < N; ++k) {
        const float x = stage_elem<ELT>(stage, full, nv, k, tid);
        c += (x > v && x > kNegInf) ? 1 : 0;
    }
    const int cnt_gt = block_sum_i(c, sm, lane, warp);
    const int take = (cnt_ge < 32 ? cnt_ge : 32);
    const int need_eq = take - cnt_gt;
    if (tid == 0) sm.red_i[0] = 0;
    cbar();
#pragma unroll 8
    for (int k = 0; k < N; ++k) {
        const float x = stage_elem<ELT>(stage, full, nv, k, tid);
        if (x > v && x > kNegInf) {
            const int pos = atomicAdd(&sm.red_i[0], 1);
            if (pos < 32) sm.cand[pos] = make_key(x, (uint32_t)(tbase + tile_elem_id<ELT>(full, k, tid)));
        }
    }
    cbar();
    // lanes equal to v, in ascending id order, until need_eq are taken
    const int NQ = full ? L::NCH : N;
    const int SPQ = full ? L::EPV : 1;
    int got = 0;
    for (int q = 0; q < NQ && got < need_eq; ++q) {
        int mine = 0;
        for (int e = 0; e < SPQ; ++e) {
            const float x = stage_elem<ELT>(stage, full, nv, q * SPQ + e, tid);
            mine += (x == v && x > kNegInf) ? 1 : 0;
        }
        int total = 0;
        int before = block_excl_scan_i(mine, &total, sm, lane, warp);
        for (int e = 0; e < SPQ; ++e) {
            const int k = q * SPQ + e;
            const float x = stage_elem<ELT>(stage, full, nv, k, tid);
            if (x == v && x > kNegInf) {
                const int pos = got + before;
                if (pos < need_eq)
                    sm.cand[cnt_gt + pos] = make_key(x, (uint32_t)(tbase + tile_elem_id<ELT>(full, k, tid)));
                ++before;
            }
        }
        got += total;
    }
    cbar();
    const int n = take;
    if (tid < n) {
        const unsigned long long key = sm.cand[tid];
        int rank = 0;
        for (int u = 0; u < n; ++u) rank += sm.cand[u] > key ? 1 : 0;
        out[rank] = key;
    }
    if (tid >= n && tid < 32) out[tid] = 0ull;
    cbar();
}

// ------------------------------------------------------------------ compute warps

// Warp-level top-4 extraction on ord32 values: returns the 4th largest
// (knocking out one lane per round), and the largest through *mx.
__device__ __forceinline__ uint32_t warp_fourth_largest(uint32_t u, int lane, uint32_t* mx) {
    uint32_t r = 0;
#pragma unroll
    for (int round = 0; round < 4; ++round) {
        r = __reduce_max_sync(kFull, u);
        if (round == 0) *mx = r;
        const unsigned b = __ballot_sync(kFull, u == r);
        if (lane == __ffs(b) - 1) u = 0u;
    }
    return r;
}

// Tile element id (within the tile) of the thread's first element equal to m.
template <int ELT>
__device__ __forceinline__ int first_equal(const unsigned char* sp, bool full, int nv, int tid, float m) {
    TileRegs<ELT> y;
    y.load(sp, full, nv, tid);
    int kf = TileRegs<ELT>::kN - 1;
#pragma unroll
    for (int k = TileRegs<ELT>::kN - 1; k >= 0; --k) kf = (y.get(k) == m) ? k : kf;
    return tile_elem_id<ELT>(full, kf, tid);
}

// Appends the keys of the thread's elements >= theta to its warp's region
// (32 keys; the counter may pass 32, which signals an overflow).  Vectors whose
// maximum is below theta are skipped after one packed compare.
template <int ELT>
__device__ __forceinline__ void append_candidates(const unsigned char* sp, int tid, float theta, int tbase,
                                                  unsigned long long* region, int* count) {
    constexpr int NCH = TileLayout<ELT>::NCH;
    constexpr int EPV = TileLayout<ELT>::EPV;
#pragma unroll 1
    for (int c = 0; c < NCH; ++c) {
        const uint4 v = lds128(sp + (size_t)(c * kConsumerThreads + tid) * 16);
        float vmax;
        if constexpr (ELT == 2) {
            const uint32_t mm = bf16x2_max(bf16x2_max(v.x, v.y), bf16x2_max(v.z, v.w));
            vmax = fmaxf(bf16_lo(mm), bf16_hi(mm));
        } else {
            vmax = fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
                         fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
        }
        if (!(vmax >= theta)) continue;
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
            const float x = (ELT == 2) ? ((e & 1) ? bf16_hi(wv[e >> 1]) : bf16_lo(wv[e >> 1])) : __uint_as_float(wv[e]);
            if (x >= theta && x > kNegInf) {
                const int pos = atomic_add_shared(count, 1);
                if (pos < 32) st_shared_u64(region + pos, make_key(x, (uint32_t)(tbase + (c * kConsumerThreads + tid) * EPV + e)));
            }
        }
    }
}

template <int ELT>
__device__ __forceinline__ void append_candidates_partial(const unsigned char* sp, int nv, int tid, float theta,
                                                          int tbase, unsigned long long* region, int* count) {
#pragma unroll 4
    for (int k = 0; k < TileLayout<ELT>::EPT; ++k) {
        const float x = stage_elem<ELT>(sp, false, nv, k, tid);
        if (x >= theta && x > kNegInf) {
            const int pos = atomic_add_shared(count, 1);
            if (pos < 32) st_shared_u64(region + pos, make_key(x, (uint32_t)(tbase + k * kConsumerThreads + tid)));
        }
    }
}

// Top-32 (descending) of the candidate regions when they hold <= 64 keys in
// total, by one warp: two 32-key bitonic sorts and a bitonic merge.
__device__ __forceinline__ unsigned long long warp_top32_of_regions(const unsigned long long* cand, const int* wcnt,
                                                                    int lane) {
    unsigned long long a = 0ull, b = 0ull;
    int before = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const int cw = wcnt[w];
        const int ia = lane - before, ib = lane + 32 - before;
        if (ia >= 0 && ia < cw) a = cand[w * 32 + ia];
        if (ib >= 0 && ib < cw) b = cand[w * 32 + ib];
        before += cw;
    }
    a = warp_sort_desc(a, lane);
    b = warp_sort_desc(b, lane);
    const unsigned long long rev = __shfl_sync(kFull, b, 31 - lane);
    return warp_bitonic_clean_desc(rev > a ? rev : a, lane);
}

template <int ELT>
__device__ __noinline__ void record_block(const Params& p, Shared& sm, int row, int entry, int chosen);

// Builds the records the merge warp queued, up to the snapshot `upto` (the
// same value in every compute thread).  Returns the new head.
template <int ELT>
__device__ __forceinline__ unsigned run_tasks(const Params& p, Shared& sm, unsigned head, unsigned upto) {
    cbar();  // the tile's readers of the candidate buffer are done (it aliases the task lists)
    while (head != upto) {
        const int4 t = sm.task[head % kTasks];
        ++head;
        record_block<ELT>(p, sm, t.x, t.z, t.y);
    }
    if (threadIdx.x == 0) vstore(&sm.task_head, head);
    return head;
}

template <int ELT>
__device__ void compute_loop(const Params& p, Shared& sm, unsigned char* stages, unsigned long long t0) {
    constexpr int S = StageCfg<ELT>::kStages;
    constexpr int TILE_BYTES = kTileBytes;
    constexpr int kTE = tile_elems<ELT>();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned long long deadline = t0 + p.timeout_ns;
    const int V = (int)p.V;
    int stage = 0, rslot = 0;
    uint32_t phase = 0, rphase = 0;
    unsigned task_head = 0;
    for (int seq = 0;; ++seq) {
        const int par = seq & 1;
        bool late = !mbar_wait(&sm.full[stage], phase, deadline);
        const int4 info = sm.info[stage];
        const bool done = info.z < 0;
        late = late || !mbar_wait(&sm.rempty[rslot], rphase ^ 1u, deadline);
        late = __any_sync(kFull, late);  // warp-uniform before any warp collective
        const unsigned char* sp = stages + (size_t)stage * TILE_BYTES;
        const int tile = info.y, mode = info.w;
        const int tbase = tile * kTE;
        const int rem = V - tbase;
        const int nv = rem < kTE ? (rem > 0 ? rem : 0) : kTE;
        const bool full = nv == kTE;
        ResultSlot& R = sm.res[rslot];
        const bool work = !late && !done;
        trace(p, kTrTileStart, info.x, tile, tid == 0 && work);

        float m = kNegInf, s = 0.0f;
        if (work) {
            // two passes over the stage: max, then sum exp(x - m); the tile is never
            // held in registers
            m = full ? stage_max<ELT>(sp, tid) : partial_max<ELT>(sp, nv, tid);
            if (mode != kModeArgmax && m > kNegInf) {
                // exp(x - m) = 2^(x*log2e - mb - mb_lo): mb_lo, the rounding residual
                // of m*log2e, is applied once, so large |m| costs no accuracy
                const float mb = m * kLog2e;
                const float mb_lo = fmaf(m, kLog2e, -mb);
                s = (full ? stage_expsum<ELT>(sp, tid, mb) : partial_expsum<ELT>(sp, nv, tid, mb)) * ex2(-mb_lo);
            }
        }
        const uint32_t om = ord32(__fadd_rn(m, 0.0f));
        if (work) {
            uint32_t omx;
            if (mode == kModeNatural) {
                // theta: min over warps of the warp's 4th largest thread maximum;
                // at least 32 lanes of the tile are >= theta
                const uint32_t o4 = warp_fourth_largest(om, lane, &omx);
                if (lane == 0) sm.wTheta[par][warp] = unord32(o4);
            } else {
                omx = __reduce_max_sync(kFull, om);
                // argmax key: smallest id among the lanes holding the warp maximum
                uint32_t id = 0xFFFFFFFFu;
                if (om == omx && m > kNegInf) id = (uint32_t)(tbase + first_equal<ELT>(sp, full, nv, tid, m));
                const uint32_t idmin = __reduce_min_sync(kFull, id);
                if (lane == 0) sm.wkey[par][warp] = ((unsigned long long)omx << 32) | (unsigned long long)(~idmin);
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.empty[stage]);  // no more reads of this stage
            }
            const float Mw = unord32(omx);
            const float sc = (m > kNegInf && mode != kModeArgmax) ? s * ex2((m - Mw) * kLog2e) : 0.0f;
            const float sw = warp_sum_f(sc);
            if (lane == 0) {
                sm.wM[par][warp] = Mw;
                sm.wS[par][warp] = sw;
            }
        }
        if (lane == 0) sm.wcnt[par][warp] = 0;
        if (tid == 0) sm.task_snap[par] = vload(&sm.task_tail);
        // B1: partials visible; every compute thread leaves together on timeout or end
        if (cbar_or(late || done)) {
            if (late) {
                if (tid == 0) atomicOr(p.status, kStatusTimeout);
            } else {
                // every record this CTA owes is queued by now (nothing is outstanding)
                task_head = run_tasks<ELT>(p, sm, task_head, sm.task_snap[par]);
                if (tid == 0) R.info = info;  // tells the merge warp to finish
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.rfull[rslot]);
            }
            return;
        }
        const unsigned task_snap = sm.task_snap[par];
        trace(p, kTrTileB1, info.x, tile, tid == 0);
        float M = sm.wM[par][0];
#pragma unroll
        for (int w = 1; w < 8; ++w) M = fmaxf(M, sm.wM[par][w]);
        if (mode == kModeNatural) {
            float theta = sm.wTheta[par][0];
#pragma unroll
            for (int w = 1; w < 8; ++w) theta = fminf(theta, sm.wTheta[par][w]);
            // candidates: each warp packs its own into cand[32*warp ..] (no atomics)
            if (m >= theta && m > kNegInf) {
                if (full) {
                    append_candidates<ELT>(sp, tid, theta, tbase, sm.cand + warp * 32, &sm.wcnt[par][warp]);
                } else {
                    append_candidates_partial<ELT>(sp, nv, tid, theta, tbase, sm.cand + warp * 32,
                                                   &sm.wcnt[par][warp]);
                }
            }
            cbar();  // B2: candidates complete
            int n = 0, over = 0;
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                const int cw = sm.wcnt[par][w];
                n += cw;
                over |= cw > 32;
            }
            trace(p, kTrTileB2, info.x, n, tid == 0);
            if (!over) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.empty[stage]);
                if (n <= 64) {
                    // one warp (rotating with the tile) sorts the <= 64 candidates
                    if (warp == (seq & 7)) R.keys[lane] = warp_top32_of_regions(sm.cand, sm.wcnt[par], lane);
                } else if (lane < sm.wcnt[par][warp]) {
                    // thread 32w+j holds candidate j of warp w; rank = # larger keys
                    const unsigned long long key = sm.cand[tid];
                    int rank = 0;
#pragma unroll 1
                    for (int w = 0; w < 8; ++w) {
                        const int cw = sm.wcnt[par][w];
                        const unsigned long long* cp = sm.cand + w * 32;
#pragma unroll 4
                        for (int u = 0; u < cw; ++u) rank += cp[u] > key ? 1 : 0;
                    }
                    if (rank < kKeysPerTile) R.keys[rank] = key;
                }
            } else {
                tile_top32_slow<ELT>(sp, full, nv, tbase, sm, R.keys);
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.empty[stage]);
            }
        } else if (tid == 0) {
            unsigned long long k0 = sm.wkey[par][0];
#pragma unroll
            for (int w = 1; w < 8; ++w) k0 = sm.wkey[par][w] > k0 ? sm.wkey[par][w] : k0;
            R.keys[0] = k0;
        }
        if (warp == 0) {
            float St = 0.0f;
            if (mode != kModeArgmax && lane < 8) {
                const float mw = sm.wM[par][lane];
                St = (mw > kNegInf) ? sm.wS[par][lane] * ex2((mw - M) * kLog2e) : 0.0f;
            }
            St += __shfl_xor_sync(kFull, St, 4);
            St += __shfl_xor_sync(kFull, St, 2);
            St += __shfl_xor_sync(kFull, St, 1);
            if (lane == 0) {
                R.info = info;
                R.M = M;
                R.S = St;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.rfull[rslot]);
        trace(p, kTrTileEnd, info.x, tile, tid == 0);
        if (task_snap != task_head) task_head = run_tasks<ELT>(p, sm, task_head, task_snap);
        if (++stage == S) {
            stage = 0;
            phase ^= 1u;
        }
        if (++rslot == kRing) {
            rslot = 0;
            rphase ^= 1u;
        }
    }
}

// ------------------------------------------------------------------ merge warp

__device__ __forceinline__ unsigned long long merge_lists(unsigned long long a, unsigned long long b, int lane) {
    const unsigned long long rev = __shfl_sync(kFull, b, 31 - lane);
    return warp_bitonic_clean_desc(rev > a ? rev : a, lane);
}

// Acceptance decision of a row whose tiles are all published (lane 0 of the
// merge warp): argmax = the row's best key; on acceptance the next row of the
// group is appended to the queue.  Returns the chosen token; *terminal is set
// when the group ends here (the caller then retires the row from
// ctrl->outstanding, after queueing its record).
__device__ __noinline__ int decide_row(const Params& p, int row, int entry, bool* requested, bool* terminal) {
    const int g = entry >> 4, j = entry & 15;
    const int4 d = __ldcg(&p.gdesc[g]);
    const int r0 = d.x, k = d.y & 0xFF, req = (d.y >> 13) & 1, samp = d.w;
    const unsigned long long bk = __ldcg(&p.row_best[row]);
    const uint32_t amax = key_id(bk);
    const int chosen = (k == 0 && samp >= 0) ? samp : (int)amax;
    const bool accept = (j < k) && (__ldg(&p.drafts[row]) == (int)amax);
    if (accept) {
        const unsigned pos = atomicAdd(&p.ctrl->q_tail, 1u);
        vstore(&p.queue[pos], queue_entry((g << 4) | (j + 1), row + 1, (d.y >> 8) & 3));
    }
    p.emitted[row] = chosen;
    if (!accept) {
        p.accepted[g] = j;
        for (int jj = j + 1; jj <= k; ++jj) p.emitted[r0 + jj] = -1;
    }
    if (req && chosen >= p.V) atomicOr(p.status, kStatusBadToken);
    *requested = req != 0;
    *terminal = !accept;
    trace(p, kTrDecision, row, accept ? 1 : 0, true);
    return chosen;
}

// Natural alternatives from the row's raw top-32 keys r (one per lane, descending),
// written into sm.rec by one warp.  Exact for the (logprob desc, id asc) order:
// see the note at the top of the file.
template <int ELT>
__device__ __noinline__ void natural_from_top32(const Params& p, int* rec, int row, long long base, int kc,
                                                float lse, unsigned long long r) {
    const int lane = threadIdx.x & 31;
    const int T = p.T;
    const bool real = r != 0ull;
    const float lp = real ? logprob(key_value(r), lse) : kNegInf;
    const int keff = (long long)kc < p.V ? kc : (int)p.V;
    const float Lk = __shfl_sync(kFull, lp, keff - 1);
    const float lp31 = __shfl_sync(kFull, lp, 31);
    bool fallback = (p.V > 32) && (lp31 == Lk);
    if (fallback) {
        // Lanes equal to Lk outside the raw top-32 lie below its 32nd key
        // (x32, id32).  If the float just below x32 already maps under Lk, they
        // all have x == x32 and ids > id32; then the top-32 suffices whenever
        // it holds at least keff - c_gt lanes equal to Lk with ids <= id32.
        const unsigned long long k32 = __shfl_sync(kFull, r, 31);
        const float x32 = key_value(k32);
        const uint32_t id32 = key_id(k32);
        if (logprob(nextafterf(x32, kNegInf), lse) != Lk) {
            const int c_above = __popc(__ballot_sync(kFull, real && lp > Lk));
            const int enough = __popc(__ballot_sync(kFull, real && lp == Lk && key_id(r) <= id32));
            if (enough >= keff - c_above) fallback = false;
        }
    }
    const unsigned long long key2 =
        real ? ((static_cast<unsigned long long>(ord32(lp)) << 32) | (r & 0xFFFFFFFFull)) : 0ull;
    const unsigned long long sorted = warp_sort_desc(key2, lane);
    const int c_gt = fallback ? __popc(__ballot_sync(kFull, real && lp > Lk)) : keff;
    if (lane < c_gt) {
        rec[2 + 2 * lane] = (int)key_id(sorted);
        rec[3 + 2 * lane] = (int)__float_as_uint(key_value(sorted));
    }
    if (fallback) {
        // lanes with logprob == Lk, smallest ids first, tile by tile; a tile can
        // hide such lanes only if its own 32nd key has logprob == Lk
        const int need = keff - c_gt;
        const unsigned lbits = __float_as_uint(Lk);
        int got = 0;
        for (int t = 0; t < T && got < need; ++t) {
            const long long t0e = (long long)t * tile_elems<ELT>();
            const long long remv = p.V - t0e;
            const int nvt = remv < tile_elems<ELT>() ? (int)remv : tile_elems<ELT>();
            const unsigned long long kmin = __ldcg(&p.part_keys[(base + t) * kKeysPerTile + 31]);
            const bool hid = nvt > 32 && kmin != 0ull && logprob(key_value(kmin), lse) == Lk;
            if (hid) {
                for (int e0 = 0; e0 < nvt && got < need; e0 += 32) {
                    const int e = e0 + lane;
                    const bool m = e < nvt && logprob(load_logit<ELT>(p, row, t0e + e), lse) == Lk;
                    const unsigned b = __ballot_sync(kFull, m);
                    const int before = __popc(b & ((1u << lane) - 1u));
                    if (m && got + before < need) {
                        rec[2 + 2 * (c_gt + got + before)] = (int)(t0e + e);
                        rec[3 + 2 * (c_gt + got + before)] = (int)lbits;
                    }
                    got += __popc(b);
                }
            } else {
                const unsigned long long key = __ldcg(&p.part_keys[(base + t) * kKeysPerTile + lane]);
                const bool m = key != 0ull && logprob(key_value(key), lse) == Lk;
                // ascending ids: sort the complements descending
                const uint32_t inv = m ? ~key_id(key) : 0u;
                const uint32_t sorted_inv = warp_sort_desc(inv, lane);
                const int cnt = __popc(__ballot_sync(kFull, m));
                if (lane < cnt && got + lane < need) {
                    rec[2 + 2 * (c_gt + got + lane)] = (int)(~sorted_inv);
                    rec[3 + 2 * (c_gt + got + lane)] = (int)lbits;
                }
                got += cnt;
            }
        }
    }
}

// Record of a requested, emitted row (whole merge warp): lse, the chosen pair,
// the natural alternatives or the explicit ids, written as 258 words.
template <int ELT>
__device__ __noinline__ void record_row(const Params& p, Shared& sm, int row, int entry, int chosen) {
    const int lane = threadIdx.x & 31;
    const int g = entry >> 4;
    const int4 d = __ldcg(&p.gdesc[g]);
    const int mode = (d.y >> 8) & 3, ids = (d.y >> 12) & 1, kc = d.z;
    const int T = p.T;
    const long long base = (long long)row * T;
    trace(p, kTrMergeStart, row, 0, lane == 0);

    // lse = M + log(sum_t s_t exp(m_t - M)); the per-tile terms are combined in
    // FP64 and the result is rounded once to FP32
    float tm = kNegInf;
    for (int t = lane; t < T; t += 32) tm = fmaxf(tm, __ldcg(&p.part_ms[base + t]).x);
    const float M = warp_max_f(tm);
    double ps = 0.0;
    for (int t = lane; t < T; t += 32) {
        const float2 ms = __ldcg(&p.part_ms[base + t]);
        ps += (double)ms.y * exp((double)ms.x - (double)M);
    }
    const double S = warp_sum_d(ps);
    const float lse = __double2float_rn((double)M + log(S));

    for (int w = lane; w < kRecordWords; w += 32) sm.mrec[w] = (w >= 2 && (w & 1) == 0) ? -1 : (int)kUnusedBits;
    __syncwarp();
    if (lane == 0) {
        sm.mrec[0] = chosen;
        sm.mrec[1] = (chosen >= 0 && chosen < p.V) ? (int)__float_as_uint(logprob(load_logit<ELT>(p, row, chosen), lse))
                                                  : (int)kUnusedBits;
        if (p.lse_out) p.lse_out[row] = lse;
    }
    if (ids) {
        int id[kMaxIds / 32];
        float xv[kMaxIds / 32];
#pragma unroll
        for (int q = 0; q < kMaxIds / 32; ++q) {
            const int i = lane + 32 * q;
            id[q] = i < kc ? __ldg(&p.token_ids[(long long)g * kMaxIds + i]) : -1;
        }
#pragma unroll
        for (int q = 0; q < kMaxIds / 32; ++q)
            xv[q] = (id[q] >= 0 && id[q] < p.V) ? load_logit<ELT>(p, row, id[q]) : 0.0f;
#pragma unroll
        for (int q = 0; q < kMaxIds / 32; ++q) {
            const int i = lane + 32 * q;
            if (i < kc) {
                int bits = (int)kUnusedBits;
                if (id[q] >= 0 && id[q] < p.V) {
                    bits = (int)__float_as_uint(logprob(xv[q], lse));
                } else {
                    atomicOr(p.status, kStatusBadId);
                }
                sm.mrec[2 + 2 * i] = id[q];
                sm.mrec[3 + 2 * i] = bits;
            }
        }
    } else if (mode == kModeNatural && kc > 0) {
        // global raw top-32: tiles merged four at a time
        const unsigned long long* kp = p.part_keys + base * kKeysPerTile + lane;
        unsigned long long r = 0;
        for (int t0 = 0; t0 < T; t0 += 4) {
            const unsigned long long a0 = __ldcg(kp + (long long)t0 * kKeysPerTile);
            const unsigned long long a1 = (t0 + 1 < T) ? __ldcg(kp + (long long)(t0 + 1) * kKeysPerTile) : 0ull;
            const unsigned long long a2 = (t0 + 2 < T) ? __ldcg(kp + (long long)(t0 + 2) * kKeysPerTile) : 0ull;
            const unsigned long long a3 = (t0 + 3 < T) ? __ldcg(kp + (long long)(t0 + 3) * kKeysPerTile) : 0ull;
            const unsigned long long b0 = merge_lists(a0, a1, lane);
            const unsigned long long b1 = merge_lists(a2, a3, lane);
            r = merge_lists(r, merge_lists(b0, b1, lane), lane);
        }
        natural_from_top32<ELT>(p, sm.mrec, row, base, kc, lse, r);
    }
    __syncwarp();
    int* out = p.records + (long long)row * kRecordWords;
    for (int w = lane; w < kRecordWords; w += 32) out[w] = sm.mrec[w];
    __syncwarp();
    trace(p, kTrMergeEnd, row, 1, lane == 0);
}

// Merges two (max, sum exp(x - max)) pairs.
__device__ __forceinline__ void ms_merge(float& m, float& s, float m2, float s2) {
    const float M = fmaxf(m, m2);
    if (M == kNegInf) return;
    s = (m > kNegInf ? s * ex2((m - M) * kLog2e) : 0.0f) + (m2 > kNegInf ? s2 * ex2((m2 - M) * kLog2e) : 0.0f);
    m = M;
}

// Record of a requested, emitted row built by the 256 compute threads (a task
// the merge warp queued after the acceptance decision): lse from the tile
// partials, the chosen pair, then the explicit-id gather or the natural
// alternatives (each warp merges every 8th tile list, warp 0 merges the 8).
// Every global load is issued before the first barrier.
template <int ELT>
__device__ __noinline__ void record_block(const Params& p, Shared& sm, int row, int entry, int chosen) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = entry >> 4;
    const int4 d = __ldcg(&p.gdesc[g]);
    const int mode = (d.y >> 8) & 3, ids = (d.y >> 12) & 1, kc = d.z;
    const int T = p.T;
    const long long base = (long long)row * T;
    const bool natural = !ids && mode == kModeNatural && kc > 0;
    trace(p, kTrMergeStart, row, 0, tid == 0);
    for (int w = tid; w < kRecordWords; w += kConsumerThreads)
        sm.rec[w] = (w >= 2 && (w & 1) == 0) ? -1 : (int)kUnusedBits;
    // loads: tile partials, the chosen logit, explicit-id logits, tile key lists
    float m = kNegInf, s = 0.0f;
    for (int t = tid; t < T; t += kConsumerThreads) {
        const float2 ms = __ldcg(&p.part_ms[base + t]);
        ms_merge(m, s, ms.x, ms.y);
    }
    float xc = 0.0f;
    if (tid == 32 && chosen >= 0 && chosen < p.V) xc = load_logit<ELT>(p, row, chosen);
    int id = -1;
    float xi = 0.0f;
    if (ids && tid < kc) {
        id = __ldg(&p.token_ids[(long long)g * kMaxIds + tid]);
        if (id >= 0 && id < p.V) xi = load_logit<ELT>(p, row, id);
    }
    if (natural) {
        const unsigned long long* kp = p.part_keys + base * kKeysPerTile + lane;
        unsigned long long r = 0;
        for (int t = warp; t < T; t += 16) {
            const unsigned long long a0 = __ldcg(kp + (long long)t * kKeysPerTile);
            const unsigned long long a1 = (t + 8 < T) ? __ldcg(kp + (long long)(t + 8) * kKeysPerTile) : 0ull;
            r = merge_lists(r, merge_lists(a0, a1, lane), lane);
        }
        sm.lists[warp][lane] = r;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(kFull, m, o), s2 = __shfl_xor_sync(kFull, s, o);
        ms_merge(m, s, m2, s2);
    }
    if (lane == 0) {
        sm.red_f[warp] = m;
        sm.red_f2[warp] = s;
    }
    if (tid == 32) sm.xchosen = xc;
    cbar();
    if (warp == 0) {
        // lse = M + log(sum_t s_t exp(m_t - M)), rounded once to FP32
        float M = sm.red_f[0], S = sm.red_f2[0];
#pragma unroll
        for (int w = 1; w < 8; ++w) ms_merge(M, S, sm.red_f[w], sm.red_f2[w]);
        float lse = 0.0f;
        if (lane == 0) lse = __double2float_rn((double)M + log((double)S));
        lse = __shfl_sync(kFull, lse, 0);
        if (lane == 0) {
            sm.lse = lse;
            sm.rec[0] = chosen;
            sm.rec[1] = (chosen >= 0 && chosen < p.V) ? (int)__float_as_uint(logprob(sm.xchosen, lse))
                                                      : (int)kUnusedBits;
            if (p.lse_out) p.lse_out[row] = lse;
        }
        if (natural) {
            const unsigned long long b0 = merge_lists(sm.lists[0][lane], sm.lists[1][lane], lane);
            const unsigned long long b1 = merge_lists(sm.lists[2][lane], sm.lists[3][lane], lane);
            const unsigned long long b2 = merge_lists(sm.lists[4][lane], sm.lists[5][lane], lane);
            const unsigned long long b3 = merge_lists(sm.lists[6][lane], sm.lists[7][lane], lane);
            const unsigned long long r = merge_lists(merge_lists(b0, b1, lane), merge_lists(b2, b3, lane), lane);
            natural_from_top32<ELT>(p, sm.rec, row, base, kc, lse, r);
        }
    }
    cbar();
    if (ids && tid < kc) {
        int bits = (int)kUnusedBits;
        if (id >= 0 && id < p.V) {
            bits = (int)__float_as_uint(logprob(xi, sm.lse));
        } else {
            atomicOr(p.status, kStatusBadId);
        }
        sm.rec[2 + 2 * tid] = id;
        sm.rec[3 + 2 * tid] = bits;
    }
    cbar();
    int* out = p.records + (long long)row * kRecordWords;
    for (int w = tid; w < kRecordWords; w += kConsumerThreads) out[w] = sm.rec[w];
    cbar();
    trace(p, kTrMergeEnd, row, 1, tid == 0);
}

// The merge warp publishes tile results to global memory and counts each
// row's finished tiles; for a row's last tile it takes the acceptance decision
// at once and queues the row's record as a task for the compute warps (or,
// when the CTA's task ring is full, writes it itself).  Results are taken in
// batches (the slots already written, up to the ring size): one fence, then
// one done-counter atomic per tile from separate lanes.
template <int ELT>
__device__ __noinline__ void merge_loop(const Params& p, Shared& sm, unsigned long long t0) {
    const int lane = threadIdx.x & 31;
    const unsigned long long deadline = t0 + p.timeout_ns;
    const int T = p.T;
    int rslot = 0;
    uint32_t rphase = 0;
    for (;;) {
        if (!mbar_wait(&sm.rfull[rslot], rphase, deadline)) {
            if (lane == 0) atomicOr(p.status, kStatusTimeout);
            return;
        }
        int n = 0;
        bool finished = false;
        do {
            const ResultSlot& R = sm.res[rslot];
            const int4 info = R.info;
            if (info.z < 0) {
                finished = true;
                break;
            }
            const int mode = info.w;
            const unsigned long long key = (mode == kModeNatural || lane == 0) ? R.keys[lane] : 0ull;
            const float Mt = R.M, St = R.S;
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&sm.rempty[rslot]);
                sm.batch[n] = make_int2(info.x, info.z);
            }
            const long long slot = (long long)info.x * T + info.y;
            if (mode == kModeNatural || lane == 0) p.part_keys[slot * kKeysPerTile + lane] = key;
            if (lane == 0) {
                p.part_ms[slot] = make_float2(Mt, St);
                atomicMax(&p.row_best[info.x], key);
            }
            trace(p, kTrPublish, info.x, info.y, lane == 0);
            ++n;
            if (++rslot == kRing) {
                rslot = 0;
                rphase ^= 1u;
            }
        } while (n < kRing && mbar_test_wait(&sm.rfull[rslot], rphase));
        __threadfence();
        __syncwarp();
        int last = 0;
        int2 b = make_int2(0, 0);
        if (lane < n) {
            b = sm.batch[lane];
            last = atomicAdd(&p.done[b.x], 1) == T - 1;
        }
        unsigned lastmask = __ballot_sync(kFull, last);
        if (lastmask) __threadfence();
        while (lastmask) {
            const int i = __ffs(lastmask) - 1;
            lastmask &= lastmask - 1;
            int4 task = make_int4(0, 0, -1, 0);
            int own = 0;  // 1: the task ring is full, the merge warp writes the record
            if (lane == 0) {
                const int2 bi = sm.batch[i];
                bool req = false, terminal = false;
                const int chosen = decide_row(p, bi.x, bi.y, &req, &terminal);
                if (req) {
                    task = make_int4(bi.x, chosen, bi.y, kModeRecord);
                    const unsigned tail = sm.task_tail;
                    if (tail - vload(&sm.task_head) < (unsigned)kTasks) {
                        sm.task[tail % kTasks] = task;
                        __threadfence_block();
                        vstore(&sm.task_tail, tail + 1u);
                    } else {
                        own = 1;
                    }
                }
                // the record is queued (or about to be written here) before the row retires
                __threadfence();
                if (terminal) atomicSub(&p.ctrl->outstanding, 1);
            }
            own = __shfl_sync(kFull, own, 0);
            if (own) {
                const int row = __shfl_sync(kFull, task.x, 0);
                const int chosen = __shfl_sync(kFull, task.y, 0);
                const int entry = __shfl_sync(kFull, task.z, 0);
                record_row<ELT>(p, sm, row, entry, chosen);
            }
        }
        if (finished) return;
    }
}

template <int ELT>
__global__ void __launch_bounds__(kThreads, StageCfg<ELT>::kMinBlocks) lp_stream_kernel(Params p) {
    constexpr int S = StageCfg<ELT>::kStages;
    constexpr int TILE_BYTES = kTileBytes;
    constexpr int kTE = tile_elems<ELT>();
    extern __shared__ __align__(16) unsigned char smem_raw[];
    unsigned char* stages = smem_raw;
    Shared& sm = *reinterpret_cast<Shared*>(smem_raw + (size_t)S * TILE_BYTES);
    const int tid = threadIdx.x;
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kConsumerThreads / 32);
        }
        for (int s = 0; s < kRing; ++s) {
            mbar_init(&sm.rfull[s], kConsumerThreads / 32);
            mbar_init(&sm.rempty[s], 1);
        }
        sm.ncand[0] = 0;
        sm.ncand[1] = 0;
        g_trace_n[0] = g_trace_n[1] = g_trace_n[2] = 0u;
        sm.task_head = 0u;
        sm.task_tail = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (vload(&p.ctrl->abort) != 0u) return;
    const unsigned long long t0 = globaltimer();
    trace(p, kTrKernel, 0, 0, tid == 0);
    const int warp = tid >> 5;
    if (warp == kConsumerThreads / 32) {
        if (tid == kConsumerThreads) producer_loop<ELT>(p, sm, stages, t0);
        return;
    }
    if (warp == kConsumerThreads / 32 + 1) {
        merge_loop<ELT>(p, sm, t0);
        return;
    }
    compute_loop<ELT>(p, sm, stages, t0);
}

template <int ELT>
constexpr int stream_smem_bytes() {
    return StageCfg<ELT>::kStages * kTileBytes + (int)sizeof(Shared);
}

}  // namespace

cudaError_t query_launch_cfg(int dtype, LaunchCfg* cfg) {
    int dev = 0, sms = 0, occ = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (dtype == 1) {
        const int smem = stream_smem_bytes<2>();
        e = cudaFuncSetAttribute(lp_stream_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, lp_stream_kernel<2>, kThreads, smem);
        cfg->smem_bytes = smem;
    } else {
        const int smem = stream_smem_bytes<4>();
        e = cudaFuncSetAttribute(lp_stream_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, lp_stream_kernel<4>, kThreads, smem);
        cfg->smem_bytes = smem;
    }
    if (e != cudaSuccess) return e;
    cfg->grid = sms * (occ > 0 ? occ : 1);
    return cudaSuccess;
}

cudaError_t launch_epilogue(const Params& p, int dtype, const LaunchCfg& cfg, cudaStream_t stream) {
    lp_prepare_kernel<<<1, 1024, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    long long work = (long long)p.rows * p.T;
    int grid = cfg.grid;
    if (work < grid) grid = work > 0 ? (int)work : 1;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(grid);
    lc.blockDim = dim3(kThreads);
    lc.dynamicSmemBytes = cfg.smem_bytes;
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    if (dtype == 1) return cudaLaunchKernelEx(&lc, lp_stream_kernel<2>, p);
    return cudaLaunchKernelEx(&lc, lp_stream_kernel<4>, p);
}

}  // namespace lp
