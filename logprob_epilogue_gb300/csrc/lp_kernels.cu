// lp_kernels.cu -- sm_103a kernels of the logprob / greedy-acceptance epilogue.
//
// Three launches per run, all on the caller's stream, each of the last two
// with programmatic dependent launch:
//
//  lp_prepare_kernel (1 CTA of 1024 threads)
//    validates group_indptr, resolves each group's request (natural
//    alternatives, explicit ids or argmax only), finishes groups that need no
//    logits, resets the per-row counters, advances the run epoch and writes
//    the depth-0 work queue: row 0 of every group that must be read.
//
//  lp_stream_kernel (persistent, 3 CTAs per SM, a few slots left to the
//  record kernel), CTAs of 10 specialised warps:
//    - producer warp (one lane): claims work items (queue position, tile) --
//      the depth-0 rows' tiles first, then rows appended after an acceptance
//      -- and streams each 32 KiB vocabulary tile (16384 BF16 or 8192 FP32
//      elements) into the CTA's stage with a TMA bulk copy (cp.async.bulk,
//      mbarrier completion, L2 evict-first);
//    - 8 compute warps: each reduces its share of a tile to its FP32 max, the
//      argmax key (atomicMax into the row's best key), the exp-sum (ex2)
//      relative to its max and, for rows that report natural alternatives, a
//      summary of its 4 largest thread maxima; the partials go to global
//      memory and the tile to the helper warp through a done slot;
//    - helper warp: counts every tile for its row and decides a row when its
//      count completes it (argmax -> greedy acceptance; on acceptance the next
//      row of the group is appended to the queue, so rows past the accepted
//      prefix are never read; a requesting row gets a record task).
//
//  lp_record_kernel (persistent, scheduled once every stream CTA has started:
//    it takes the slots the stream grid leaves and those of stream CTAs that
//    exit): claims record tasks as the deciders append them and builds each
//    record while the stream kernel runs -- lse = M + log(sum s_t exp(m_t -
//    M)) from the tile partials, the chosen token's logprob, the top-K
//    natural alternatives or the explicit-id gather, the 258-word record.
//
// Sources: "logprobs-design.md" (generation-logprob contract; the four-launch
// reduction paragraph: FP32 tile maxima and exponential sums, a per-position
// normalisation, best-32 integer sort keys over reported FP32 logprobs and
// inverse ids, ties from the subtraction included, equal values at the cutoff
// taking the smallest ids, signed zero normalised, padded lanes excluded,
// explicit ids gathered from raw logits) and "mtp-design.md" ("A speculative
// round is a state transaction", steps 2-3).
//
// Exactness of the natural alternatives (natural_record): fl32(x - lse) is
// non-decreasing in x, so a candidate set holding every lane >= a threshold
// theta with at least 32 lanes above it holds the row's best K by logprob,
// except lanes below theta that tie with the K-th value after the
// subtraction; those exist only if the float just below theta already reports
// that value, and are then collected in id order.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "lp_internal.h"

namespace lp {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kPosInf = __builtin_huge_valf();
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

template <typename T>
__device__ __forceinline__ T vload(const T* p) { return *reinterpret_cast<const volatile T*>(p); }
template <typename T>
__device__ __forceinline__ void vstore(T* p, T v) { *reinterpret_cast<volatile T*>(p) = v; }

// Run-tagged words: epoch << 32 | payload.  The tile partials and record tasks
// that the record kernel reads while the stream kernel still runs are written
// as pairs of such words with relaxed 64-bit stores (each word is single-copy
// atomic), and a reader takes a pair only once both words carry the run's
// epoch: a word still in flight, or left by an earlier run, is never mistaken
// for this run's.
__device__ __forceinline__ unsigned long long tagged(uint32_t ep, uint32_t v) {
    return ((unsigned long long)ep << 32) | (unsigned long long)v;
}
__device__ __forceinline__ bool has_epoch(const ulonglong2& w, uint32_t ep) {
    return (uint32_t)(w.x >> 32) == ep && (uint32_t)(w.y >> 32) == ep;
}
__device__ __forceinline__ void st_tagged(ulonglong2* p, unsigned long long a, unsigned long long b) {
    asm volatile("st.relaxed.gpu.global.v2.b64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}
__device__ __forceinline__ ulonglong2 ld_tagged(const ulonglong2* p) {
    ulonglong2 v;
    asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(v.x), "=l"(v.y) : "l"(p) : "memory");
    return v;
}

// ---- optional device timeline (plans created with the trace flag)
//
// Each CTA has three event rings (producer, compute, merge warp) of
// p.trace_cap events; an event is (globaltimer ns, type << 56 | row << 24 | tile).
enum : unsigned { kTrKernel = 1, kTrClaim, kTrIssue, kTrTileStart, kTrTileEnd, kTrPublish, kTrMergeStart,
                  kTrDecision, kTrMergeEnd, kTrPrepStart, kTrPrepEnd, kTrExit, kTrTileB1, kTrTileB2,
                  kTrWarpAppend, kTrWarpDone, kTrRecStart, kTrRecEnd, kTrRecA, kTrRecB, kTrRecC, kTrRecD };

__shared__ unsigned g_trace_n[kTraceRoles];  // per-CTA event counts (producer, compute, merge, record)

__device__ __forceinline__ void trace(const Params& p, unsigned type, int row, int tile, bool writer) {
    if (p.trace == nullptr || !writer) return;
    const int role = type == kTrClaim || type == kTrIssue || type == kTrExit ? 0
                   : (type == kTrTileStart || type == kTrTileEnd || type == kTrKernel || type == kTrTileB1 ||
                      type == kTrTileB2 || type == kTrWarpAppend || type == kTrWarpDone) ? 1 : 2;
    unsigned* cnt = g_trace_n + role;
    const unsigned i = atomicAdd(cnt, 1u);  // several warps may record into one ring
    if (i >= (unsigned)p.trace_cap) return;
    atomicMax(&p.trace_count[blockIdx.x * kTraceRoles + role], i + 1);
    unsigned long long* e = p.trace + (((size_t)blockIdx.x * kTraceRoles + role) * p.trace_cap + i) * 2;
    e[0] = globaltimer();
    e[1] = ((unsigned long long)type << 56) | ((unsigned long long)(row & 0xFFFFFFFF) << 24) |
           (unsigned long long)(tile & 0xFFFFFF);
}

// Record-kernel events go to the record-role ring of CTA blockIdx.x.
__device__ __forceinline__ void rtrace(const Params& p, unsigned type, int row) {
    if (p.trace == nullptr || threadIdx.x != 0 || (int)blockIdx.x >= p.trace_ctas) return;
    const unsigned i = g_trace_n[3]++;  // thread 0 alone records: no round trip on the record's path
    if (i >= (unsigned)p.trace_cap) return;
    atomicMax(&p.trace_count[blockIdx.x * kTraceRoles + 3], i + 1);
    unsigned long long* e = p.trace + (((size_t)blockIdx.x * kTraceRoles + 3) * p.trace_cap + i) * 2;
    e[0] = globaltimer();
    e[1] = ((unsigned long long)type << 56) | ((unsigned long long)(row & 0xFFFFFFFF) << 24);
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

#ifndef LP_NATURAL_KEEP
#define LP_NATURAL_KEEP 0
#endif
__device__ __forceinline__ uint64_t evict_normal_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
    return pol;
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

__device__ __forceinline__ float warp_min_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
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
template <typename T>
__device__ __forceinline__ T warp_bitonic_clean_desc(T v, int lane) {
#pragma unroll
    for (int j = 16; j > 0; j >>= 1) {
        const T p = __shfl_xor_sync(kFull, v, j);
        const bool lower = (lane & j) == 0;
        v = lower ? (p > v ? p : v) : (p < v ? p : v);
    }
    return v;
}

constexpr int kMaxStages = 8;
constexpr int kWarps = kConsumerThreads / 32;  // compute warps
static_assert(StageCfg<2>::kStages <= kMaxStages && StageCfg<4>::kStages <= kMaxStages, "stage count");

// Tiles handed from the compute warps to the helper warp, in order.
constexpr int kDoneRing = 4;

#ifndef LP_STAGE_ALIGN
#define LP_STAGE_ALIGN 128
#endif
constexpr uint32_t kStageAlign = LP_STAGE_ALIGN < 16 ? 16u : (uint32_t)LP_STAGE_ALIGN;

struct Shared {
    uint64_t full[kMaxStages];       // stage filled (producer + TMA)
    uint64_t empty[kMaxStages];      // stage released (8 compute warps)
    uint64_t dfull[kDoneRing];       // done slot: the 8 compute warps finished the tile
    uint64_t dfree[kDoneRing];       // done slot: read by the helper warp
    int4 dslot[kDoneRing];           // done slot: (row, queue entry, 0, 0) of the tile
    int sel_exit;                    // compute warps that have finished (the helper stops at 8)
    unsigned long long wbest[kWarps];  // each warp's last atomic results (an issue dependency)
    int4 info[kMaxStages];           // work item of each stage
};

// Natural alternatives in the record stage (see natural_record).
constexpr int kCandThreads = 512;    // candidate thread slots (tile << 8 | thread)
constexpr int kCandShares = 16;      // warp shares re-read whole (their 4th summary entry reaches theta)
constexpr int kCandKeys = 1024;      // candidate logprob keys

// Shared memory of the record kernel.
struct RecShared {
    float red_f[kWarps];
    float red_f2[kWarps];
    int red_i[kWarps];
    int red_x[kWarps];                      // natural_exact: counts
    float lse;
    float xchosen;
    float xlim;                             // prompt scoring: largest logit whose lp is the target's
    int corr;                               // prompt scoring: logits in (target's, xlim]
    uint32_t theta_o;                       // natural: ord32 of the candidate threshold (0: none)
    int slow;                               // natural: some candidate thread was not prefetched
    uint32_t wtop[kWarps][8];               // natural: each warp's 8 largest summary entry values
    unsigned long long wsel[kWarps][8];     // natural: those entries (record fast path)
    unsigned long long lkey;                // natural: the keff-th best logprob key
    int n_thr, n_sh, n_keys;                // natural: candidate threads, shares and keys
    int rec[kRecordWords + 2];              // record being assembled
    uint32_t cthr[kCandThreads];
    uint32_t csh[kCandShares];
    alignas(16) unsigned long long ckeys[kCandKeys + 8];
};

// ---- tile element access
//
// Thread i owns the 16-byte vectors c*256 + i (c = 0..NCH-1), so element
// k = c*EPV + s of the thread is tile element (c*256 + i)*EPV + s.  The last,
// partial tile of a row is read the same way once its lanes past V are set to
// -inf in the stage (fill_partial).

template <int ELT>
struct TileLayout {
    static constexpr int EPV = 16 / ELT;          // elements per 16-byte vector
    static constexpr int NCH = kTileBytes / 16 / kConsumerThreads;  // vectors per thread (8)
};

// 16-byte shared-memory load through an explicit shared-space address.
__device__ __forceinline__ uint4 lds128(const void* p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_u32(p)));
    return v;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Streaming passes over a full stage (thread i reads vectors c*256 + i).
//
// Pass 1 keeps the maximum of each of the thread's 16-byte vectors in cm[c]
// (BF16: packed bf16x2, the even elements' maximum in the low half, the odd
// ones' in the high half; FP32: the float bits), so that the argmax search and
// the candidate selection later touch only the vectors that can matter.
template <int ELT>
__device__ __forceinline__ float vec_max(uint32_t cm) {
    if constexpr (ELT == 2) {
        return fmaxf(bf16_lo(cm), bf16_hi(cm));
    } else {
        return __uint_as_float(cm);
    }
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Vector c of the calling thread (16 bytes) from the stage.  A partial tile
// (FULL = false) has had every lane past nv set to -inf in the stage first
// (fill_partial), so both read the same way.
template <int ELT, bool FULL>
__device__ __forceinline__ uint4 ld_vec(const unsigned char* sp, int c, int tid, int nv) {
    return lds128(sp + (size_t)(c * kConsumerThreads + tid) * 16);
}

// Sets the lanes past nv of the calling thread's vectors to -inf, in the stage:
// the last tile of a row is then read like a full one.  A thread touches only
// its own vectors, the ones it reads later, so no barrier is needed; the proxy
// fence before the stage is released (tile_work) orders these writes before
// the next bulk copy into the stage.
template <int ELT>
__device__ __forceinline__ void fill_partial(unsigned char* sp, int tid, int nv) {
    constexpr int EPV = 16 / ELT;
    constexpr uint32_t kNegInfW = ELT == 2 ? 0xFF80FF80u : 0xFF800000u;
#pragma unroll
    for (int c = 0; c < TileLayout<ELT>::NCH; ++c) {
        const int v = c * kConsumerThreads + tid;
        const int valid = nv - v * EPV;
        if (valid >= EPV) continue;
        uint4* dst = reinterpret_cast<uint4*>(sp + (size_t)v * 16);
        if (valid <= 0) {
            *dst = make_uint4(kNegInfW, kNegInfW, kNegInfW, kNegInfW);
            continue;
        }
        const uint4 x = lds128(dst);
        uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if constexpr (ELT == 2) {
                if (2 * i >= valid) w[i] = kNegInfW;
                else if (2 * i + 1 >= valid) w[i] = (w[i] & 0xFFFFu) | 0xFF800000u;
            } else {
                if (i >= valid) w[i] = kNegInfW;
            }
        }
        *dst = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

template <int ELT, bool FULL>
__device__ __forceinline__ float stage_max(const unsigned char* sp, int tid, int nv,
                                           uint32_t (&cm)[TileLayout<ELT>::NCH]) {
    constexpr int NCH = TileLayout<ELT>::NCH;
    if constexpr (ELT == 2) {
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const uint4 v = ld_vec<ELT, FULL>(sp, c, tid, nv);
            cm[c] = bf16x2_max(bf16x2_max(v.x, v.y), bf16x2_max(v.z, v.w));
        }
        uint32_t a = cm[0], b = cm[1];
#pragma unroll
        for (int c = 2; c < NCH; c += 2) {
            a = bf16x2_max(a, cm[c]);
            b = bf16x2_max(b, cm[c + 1]);
        }
        a = bf16x2_max(a, b);
        return fmaxf(bf16_lo(a), bf16_hi(a));
    } else {
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const uint4 v = ld_vec<ELT, FULL>(sp, c, tid, nv);
            cm[c] = __float_as_uint(fmax3(__uint_as_float(v.x), __uint_as_float(v.y),
                                          fmaxf(__uint_as_float(v.z), __uint_as_float(v.w))));
        }
        float a = __uint_as_float(cm[0]), b = __uint_as_float(cm[1]);
#pragma unroll
        for (int c = 2; c < NCH; c += 2) {
            a = fmaxf(a, __uint_as_float(cm[c]));
            b = fmaxf(b, __uint_as_float(cm[c + 1]));
        }
        return fmaxf(a, b);
    }
}

// Packed FP32 pairs (two lanes of work per instruction on the FMA pipe).
__device__ __forceinline__ unsigned long long f2_pack(float lo, float hi) {
    return (static_cast<unsigned long long>(__float_as_uint(hi)) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long f2_ex2(unsigned long long a) {
    return f2_pack(ex2(__uint_as_float(static_cast<uint32_t>(a))), ex2(__uint_as_float(static_cast<uint32_t>(a >> 32))));
}
__device__ __forceinline__ float f2_sum(unsigned long long a) {
    return __uint_as_float(static_cast<uint32_t>(a)) + __uint_as_float(static_cast<uint32_t>(a >> 32));
}

// Pass 2: sum of 2^(x*log2e - mb) over the thread's elements, two at a time
// (-inf elements contribute 0).
template <int ELT, bool FULL>
__device__ __forceinline__ float stage_expsum(const unsigned char* sp, int tid, int nv, float mb) {
    constexpr int NCH = TileLayout<ELT>::NCH;
    const unsigned long long L2E = f2_pack(kLog2e, kLog2e), NMB = f2_pack(-mb, -mb);
    unsigned long long s0 = 0ull, s1 = 0ull;  // two accumulators: the vector maxima stay live
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
        const uint4 v = ld_vec<ELT, FULL>(sp, c, tid, nv);
        if constexpr (ELT == 2) {
            s0 = f2_add(s0, f2_ex2(f2_fma(f2_pack(bf16_lo(v.x), bf16_hi(v.x)), L2E, NMB)));
            s1 = f2_add(s1, f2_ex2(f2_fma(f2_pack(bf16_lo(v.y), bf16_hi(v.y)), L2E, NMB)));
            s0 = f2_add(s0, f2_ex2(f2_fma(f2_pack(bf16_lo(v.z), bf16_hi(v.z)), L2E, NMB)));
            s1 = f2_add(s1, f2_ex2(f2_fma(f2_pack(bf16_lo(v.w), bf16_hi(v.w)), L2E, NMB)));
        } else {
            const unsigned long long a = (static_cast<unsigned long long>(v.y) << 32) | v.x;
            const unsigned long long b = (static_cast<unsigned long long>(v.w) << 32) | v.z;
            s0 = f2_add(s0, f2_ex2(f2_fma(a, L2E, NMB)));
            s1 = f2_add(s1, f2_ex2(f2_fma(b, L2E, NMB)));
        }
    }
    return f2_sum(f2_add(s0, s1));
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
// Entry flags.  kEntryNext: the group has a row after this one (a read-ahead
// candidate).  Chained entries only: kEntryShared, the row's tiles are claimed
// through tclaim (read-ahead had started on it); kEntrySkip, read-ahead had
// claimed all of them (nothing to take).
constexpr unsigned long long kEntryShared = 1ull << 30;
constexpr unsigned long long kEntrySkip = 1ull << 31;
constexpr unsigned long long kEntryNext = 1ull << 62;
__device__ __forceinline__ int entry_gj(unsigned long long e) { return (int)((e >> 32) & 0x3FFFFFFFu); }

// ------------------------------------------------------------------ prepare

// Inputs of one group, loaded together (one memory round trip).
struct GroupIn {
    int r0, r1, req, samp, cnt, K;
};

__device__ __forceinline__ GroupIn load_group(const Params& p, int g) {
    GroupIn x;
    if (p.targets != nullptr) {  // prompt scoring: row g alone, 20 natural alternatives, chosen = target
        x.r0 = g;
        x.r1 = g + 1;
        x.req = 1;
        x.samp = __ldg(&p.targets[g]);
        x.cnt = 0;
        x.K = kScoreAlts;
        return x;
    }
    x.r0 = __ldg(&p.indptr[g]);
    x.r1 = __ldg(&p.indptr[g + 1]);
    x.req = __ldg(&p.requested[g]);
    x.samp = __ldg(&p.sampled[g]);
    x.cnt = __ldg(&p.id_counts[g]);
    x.K = __ldg(&p.top_k[g]);
    return x;
}

// Waves of first claims whose tiles the stream kernel brings into L2 before
// its dependent-launch wait (0: none).
#ifndef LP_EARLY_PREFETCH
#define LP_EARLY_PREFETCH 1
#endif
#ifndef LP_PREP_THREADS
#define LP_PREP_THREADS 1024
#endif
__global__ void __launch_bounds__(LP_PREP_THREADS) lp_prepare_kernel(Params p) {
    asm volatile("griddepcontrol.launch_dependents;");
    if (p.trace != nullptr && threadIdx.x == 0) {
        unsigned long long* e = p.trace + ((size_t)p.trace_ctas * kTraceRoles) * p.trace_cap * 2;
        e[0] = globaltimer();
        e[1] = (unsigned long long)kTrPrepStart << 56;
        e[4] = ~0ull;  // first record-kernel start (atomicMin)
        e[5] = (unsigned long long)kTrRecStart << 56;
        e[6] = 0ull;   // last record-kernel end (atomicMax)
        e[7] = (unsigned long long)kTrRecEnd << 56;
    }
    if (threadIdx.x == 0) {
        // the run's epoch: never 0 (zeroed scratch) nor all ones (poisoned scratch)
        unsigned ep = p.ctrl->epoch + 1u;
        if (ep == 0xFFFFFFFFu || ep == 0u) ep = 1u;
        p.ctrl->epoch = ep;
    }
    __shared__ int s_warp[32];
    __shared__ int s_total;
    __shared__ int s_base;
    __shared__ unsigned s_chain;  // drafts of the groups that are read: the most rows acceptances can append
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int G = p.G;
    const int nthr = blockDim.x;
    // this thread's first group: its inputs are in flight while the rows are reset
    GroupIn in0 = {0, 1, 0, 0, 0, 0};
    if (tid < G) in0 = load_group(p, tid);
    // the deciders read drafts (and EOS tokens) on the verify chains' path:
    // bring them into L2 now
    if (p.drafts != nullptr)
        for (int r = tid * 32; r < p.rows; r += nthr * 32) asm volatile("prefetch.global.L2 [%0];" ::"l"(p.drafts + r));
    if (p.eos != nullptr)
        for (int g = tid * 32; g < G; g += nthr * 32) asm volatile("prefetch.global.L2 [%0];" ::"l"(p.eos + g));
    for (int r = tid; r < p.rows; r += nthr) {
        p.done[r] = 0;
        p.queue[r] = ~0ull;
        p.tclaim[r] = 0u;
        p.row_best[r] = 0ull;
    }
    if (tid == 0) *p.status = 0u;
    // validation: indptr starts at >= 0, ends at <= rows, group sizes 1..k_max+1
    int ok = 1;
    for (int g = tid; g < G; g += nthr) {
        const GroupIn x = g == tid ? in0 : load_group(p, g);
        if (x.r1 - x.r0 < 1 || x.r1 - x.r0 - 1 > p.k_max) ok = 0;
        if (g == 0 && x.r0 < 0) ok = 0;
        if (g == G - 1 && x.r1 > p.rows) ok = 0;
    }
    ok = __syncthreads_and(ok);
    if (!ok) {
        if (tid == 0) {
            atomicOr(p.status, kStatusBadGroup);
            p.ctrl->abort = 1u;
            p.ctrl->fresh_next = 0u;
            p.ctrl->chain_next = 0u;
            p.ctrl->chain_tail = 0u;
            p.ctrl->fresh_rows = 0u;
            p.ctrl->chain_max = 0u;
            p.ctrl->outstanding = 0;
            p.ctrl->rec_count = 0u;
            p.ctrl->rec_claim = 0u;
            p.ctrl->retired = 0u;
        }
        return;
    }
    if (tid == 0) {
        s_base = 0;
        s_chain = 0u;
    }
    __syncthreads();
    // without read-ahead a row is decided when its tiles are counted; with it,
    // also only once its parent accepted (depth-0 rows: from the start)
    const int parent_bias = p.read_ahead ? kParentDone : 0;
    unsigned st = 0;
    for (int g0 = 0; g0 < G; g0 += nthr) {
        const int g = g0 + tid;
        int need = 0, row0 = 0, mode0 = 0, k0 = 0;
        if (g < G) {
            const GroupIn x = g0 == 0 ? in0 : load_group(p, g);
            const int r0 = x.r0;
            int k = x.r1 - r0 - 1;
            const int req = x.req != 0;
            int samp = x.samp;
            // commit clipping at the output budget: at most `budget` tokens, so
            // rows past budget - 1 are never read; <= 0: the request is at its
            // limit and takes no step
            const int budget = p.budget != nullptr ? __ldg(&p.budget[g]) : 0x7FFFFFFF;
            const bool at_limit = budget <= 0;
            if (!at_limit && k > budget - 1) {
                for (int jj = budget; jj <= k; ++jj) p.emitted[r0 + jj] = -1;
                k = budget - 1;
                samp = -1;  // a verify group's target row stays greedy when clipped to it
            }
            int cnt = x.cnt;
            int K = x.K;
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
                    // the record gathers these ids at the end of the run: bring them into L2 now
                    const int* tp = p.token_ids + (long long)g * kMaxIds;
                    for (int b = 0; b < cnt; b += 32) asm volatile("prefetch.global.L2 [%0];" ::"l"(tp + b));
                } else {
                    if ((K < 0 || K > p.k_alt_max) && p.targets == nullptr) {
                        st |= kStatusBadCount;
                        K = K < 0 ? 0 : p.k_alt_max;
                    }
                    kc = K;
                    mode = K > 0 ? kModeNatural : kModeLse;
                }
            }
            need = req || k >= 1 || samp < 0;
            if (at_limit) {
                need = 0;
                for (int jj = 0; jj <= k; ++jj) p.emitted[r0 + jj] = -1;
                p.accepted[g] = -1;
            } else if (p.targets != nullptr) {
                // prompt scoring: a row without a valid target is not read; its
                // record is the invalid one (id -1, NaN, rank 0, ids -1)
                need = samp >= 0 && samp < p.V;
                if (!need) {
                    if (samp >= p.V) st |= kStatusBadToken;
                    int* rec = p.score_records + (long long)r0 * kScoreWords;
                    rec[0] = -1;
                    rec[1] = (int)kUnusedBits;
                    rec[2] = 0;
                    for (int i = 0; i < kScoreAlts; ++i) {
                        rec[3 + 2 * i] = -1;
                        rec[4 + 2 * i] = (int)kUnusedBits;
                    }
                }
            } else if (!need) {
                if (samp >= p.V) st |= kStatusBadToken;
                p.emitted[r0] = samp;
                p.accepted[g] = 0;
            }
            p.gdesc[g] = make_int4(r0, k | (mode << 8) | (ids << 12) | (req << 13), kc, samp);
            row0 = r0;
            mode0 = mode;
            k0 = k;
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
        if (need) {
            const int qpos = s_base + s_warp[warp] + pos_in_warp;
            p.queue[qpos] = queue_entry(g << 4, row0, mode0) | (k0 >= 1 ? kEntryNext : 0ull);
            p.done[row0] = parent_bias;
            if (k0 > 0) atomicAdd(&s_chain, (unsigned)k0);
        }
        __syncthreads();
        if (tid == 0) s_base += s_total;
        __syncthreads();
    }
    if (st) atomicOr(p.status, st);
    if (p.trace != nullptr) {
        for (int i = tid; i < p.trace_ctas * kTraceRoles; i += nthr) p.trace_count[i] = 0u;
    }
    if (tid == 0) {
        if (p.trace != nullptr) {
            unsigned long long* e = p.trace + ((size_t)p.trace_ctas * kTraceRoles) * p.trace_cap * 2;
            e[2] = globaltimer();
            e[3] = (unsigned long long)kTrPrepEnd << 56;
        }
        p.ctrl->fresh_next = 0u;
        p.ctrl->chain_next = 0u;
        p.ctrl->chain_tail = 0u;
        p.ctrl->fresh_rows = static_cast<unsigned>(s_base);
        p.ctrl->chain_max = s_chain;
        p.ctrl->outstanding = s_base;
        p.ctrl->rec_count = 0u;
        p.ctrl->rec_claim = 0u;
        p.ctrl->retired = 0u;
        p.ctrl->abort = 0u;
    }
}

// ------------------------------------------------------------------ producer
//
// One lane draws work items one at a time and streams each 32 KiB tile into a
// shared-memory stage with a TMA bulk copy.  Fresh items (tiles of the depth-0
// rows, the roots of every verify chain) come first, claimed one ahead with
// their queue entries prefetched, so all chains start as early as the
// bandwidth allows.  Then come chained items (rows appended after an
// acceptance): each producer owns the next chained item it claimed (claims
// run ahead of the appended rows, in order) and takes it as soon as the queue
// entry of its row is published.  Single-item claims spread a row's tiles over
// many CTAs.
constexpr unsigned kNone = 0xFFFFFFFFu;
// Stream-CTA slots of the device left to the record kernel from the start of a run.
#ifndef LP_RECORD_SLOTS
#define LP_RECORD_SLOTS 24
#endif
// 0: stream CTAs exit only when no chained item can come; k > 0: also when the
// waiting chained claims cover k/4 of the next row of every outstanding group.
#ifndef LP_SURPLUS_EXIT
#define LP_SURPLUS_EXIT 0
#endif
// A producer with no claim retires its CTA when at least this many appended
// record tasks wait unclaimed (0: never), up to 1/LP_RETIRE_SHARE of the grid:
// the slot goes to a record CTA, so that the records keep pace with the
// decisions instead of piling up behind the last one.
#ifndef LP_RETIRE_BACKLOG
#define LP_RETIRE_BACKLOG 16
#endif
#ifndef LP_RETIRE_SHARE
#define LP_RETIRE_SHARE 4
#endif
// A producer reads ahead only after waiting this long for a chained item.
#ifndef LP_READ_AHEAD_IDLE_NS
#define LP_READ_AHEAD_IDLE_NS 1000
#endif
constexpr unsigned long long kReadAheadIdleNs = LP_READ_AHEAD_IDLE_NS;

// The producer warp's lanes load the first queue entries beside the producer
// lane's first claim (LP_QUEUE_WINDOW): a run's first items come from the
// first rows of the queue, so the claim's entry is then known one round trip
// sooner.
#ifndef LP_QUEUE_WINDOW
#define LP_QUEUE_WINDOW 1
#endif

// First claim of a producer: its fresh ticket, the run's fresh-row and
// chained-row counts, and the ticket's queue entry when the window held it
// (else all ones: to be loaded).
struct FirstClaim {
    unsigned ticket, F, CM;
    unsigned long long entry;
};

__device__ __forceinline__ FirstClaim first_claim(const Params& p) {
    const int lane = threadIdx.x & 31;
    Ctrl* ctrl = p.ctrl;
    FirstClaim f = {0u, 0u, 0u, ~0ull};
    unsigned long long qe = ~0ull;
    if (LP_QUEUE_WINDOW && lane < p.rows) qe = vload(&p.queue[lane]);
    if (lane == 0) {
        f.ticket = atomicAdd(&ctrl->fresh_next, 1u);
        f.F = vload(&ctrl->fresh_rows);
        f.CM = vload(&ctrl->chain_max);
    }
    f.ticket = __shfl_sync(kFull, f.ticket, 0);
    f.F = __shfl_sync(kFull, f.F, 0);
    const unsigned pos = f.ticket / (unsigned)p.T;
    const unsigned long long e = __shfl_sync(kFull, qe, (int)(pos & 31u));
    if (LP_QUEUE_WINDOW && pos < 32u && pos < f.F) f.entry = e;
    return f;
}

template <int ELT>
__device__ __noinline__ void producer_loop(const Params& p, Shared& sm, unsigned char* stages, unsigned long long t0,
                                           FirstClaim first) {
    constexpr int S = StageCfg<ELT>::kStages;
    constexpr int kTE = tile_elems<ELT>();
    const unsigned long long deadline = t0 + p.timeout_ns;
    const uint64_t policy = evict_first_policy();
    const uint64_t npolicy = LP_NATURAL_KEEP ? evict_normal_policy() : policy;
    Ctrl* ctrl = p.ctrl;
    const unsigned T = (unsigned)p.T;
    // Every item, the first included, is claimed through a counter: a CTA
    // that is not resident holds no work, so the run never waits for one (the
    // grid need not be co-resident, e.g. beside another kernel).  The first
    // chained claim waits until the first copy is issued.
    unsigned chain_claim = kNone;
    unsigned long long ra_e = ~0ull;  // read-ahead candidate: entry of the successor of the last row streamed
    unsigned long long idle_t0 = 0;   // start of the current wait for a chained item (0: not waiting)
    unsigned fresh_ahead = first.ticket;
    const unsigned F = first.F;
    const unsigned CM = first.CM;
    const unsigned fresh_items = F * T;
    // A chained claim at or past CM rows can never be taken (no more rows can
    // be appended): once this producer holds one it has no work left, and
    // (without read-ahead) its CTA exits, which leaves the multiprocessor to
    // the record kernel.
    bool fresh_done = fresh_ahead >= fresh_items;
    bool chains_over = false;
    // Retiring early (LP_SURPLUS_EXIT): a producer whose last poll found the
    // chained claims already waiting to cover the next row of every outstanding
    // group (scaled) takes no new claim, and its CTA exits.
    bool surplus = false;
    auto claim_chain = [&]() {
        if (LP_SURPLUS_EXIT && surplus && fresh_done && !p.read_ahead) {
            chains_over = true;
            return;
        }
        // record pressure: record tasks wait with no record CTA to take them;
        // a producer without a claim leaves its slot to the record kernel
        // (at most a share of the grid does)
        if (LP_RETIRE_BACKLOG > 0 && fresh_done && p.build_records && !p.read_ahead) {
            const int backlog = (int)(vload(&ctrl->rec_count) - vload(&ctrl->rec_claim));
            if (backlog >= LP_RETIRE_BACKLOG &&
                atomicAdd(&ctrl->retired, 1u) < (unsigned)(p.stream_grid / LP_RETIRE_SHARE)) {
                chains_over = true;
                return;
            }
        }
        chain_claim = atomicAdd(&ctrl->chain_next, 1u);
        if (chain_claim / T >= CM) {
            chain_claim = kNone;
            chains_over = true;
        }
    };
    unsigned long long fresh_entry =
        fresh_done ? ~0ull : ((long long)first.entry >= 0 ? first.entry : vload(&p.queue[fresh_ahead / T]));
    int stage = 0;
    uint32_t phase = 0;
    bool timed_out = false;
    for (;;) {
        int4 item = make_int4(0, 0, -1, 0);
        if (p.debug_flags & kDebugForceTimeout) {
            // Test hook: wait on a flag that nothing sets, until the limit.
            while (vload(&ctrl->never) == 0u) {
                if (globaltimer() > deadline) break;
                __nanosleep(1000);
            }
            timed_out = true;
        } else {
            unsigned long long e = ~0ull;
            unsigned tile = 0;
            for (;;) {
                if (!fresh_done && fresh_ahead != kNone) {
                    e = fresh_entry;
                    tile = fresh_ahead % T;
                    fresh_ahead = kNone;  // the next one is claimed once this copy is issued
                    break;
                }
                // this poll's loads, issued together: the chained item's entry
                // and the outstanding groups
                const unsigned cpos = chain_claim == kNone ? kNone : F + chain_claim / T;
                unsigned long long ce = ~0ull;
                if (cpos < (unsigned)p.rows) ce = vload(&p.queue[cpos]);
                const int out = fresh_done ? vload(&ctrl->outstanding) : 1;
                if (LP_SURPLUS_EXIT && fresh_done) {
                    const long long waiting = (long long)vload(&ctrl->chain_next) - (long long)vload(&ctrl->chain_tail) * T;
                    surplus = waiting * 4 >= (long long)(out > 0 ? out : 0) * T * LP_SURPLUS_EXIT;
                }
                // the chained item, once the queue entry of its row is published
                if ((long long)ce >= 0) {
                    e = ce;
                    if (e & kEntrySkip) {  // read-ahead claimed every tile of the row
                        chain_claim = kNone;
                        e = ~0ull;
                    } else if (e & kEntryShared) {  // read-ahead claimed some: take the next one
                        chain_claim = kNone;
                        const unsigned v = atomicAdd(&p.tclaim[e & 0x0FFFFFFFu], 1u);
                        if (v < T) {
                            tile = v;
                            break;
                        }
                        e = ~0ull;
                    } else {
                        tile = chain_claim % T;
                        chain_claim = kNone;
                        break;
                    }
                }
                if (!fresh_done) {
                    fresh_ahead = atomicAdd(&ctrl->fresh_next, 1u);
                    fresh_done = fresh_ahead >= fresh_items;
                    if (!fresh_done) fresh_entry = vload(&p.queue[fresh_ahead / T]);
                    continue;
                }
                if (chain_claim == kNone && !chains_over) {
                    claim_chain();
                    continue;
                }
                if (chains_over && !p.read_ahead) {
                    e = ~0ull;
                    break;
                }
                // nothing to take yet.  After a while without chained items
                // (their queue has run dry, the verify chains are the work
                // left) and with a stage free, read ahead: a tile of the
                // successor of the last row streamed, not decided yet
                const unsigned long long now = globaltimer();
                if (idle_t0 == 0) idle_t0 = now;
                if ((long long)ra_e >= 0 && now - idle_t0 > kReadAheadIdleNs &&
                    mbar_test_wait(&sm.empty[stage], phase ^ 1u)) {
                    const unsigned v = atomicAdd(&p.tclaim[ra_e & 0x0FFFFFFFu], 1u);
                    const unsigned long long se = ra_e;
                    if (v >= T - 1) ra_e = ~0ull;  // no tile of it left after this claim (or closed)
                    if (v < T) {
                        e = se;
                        tile = v;
                        break;
                    }
                }
                // the run is complete once no group is outstanding
                if (out <= 0) {
                    __threadfence();
                    // final once nothing is outstanding: a claim below it has its entry published
                    if (chain_claim / T < vload(&ctrl->chain_tail)) continue;
                    e = ~0ull;
                    break;
                }
                if (now > deadline) {
                    timed_out = true;
                    e = ~0ull;
                    break;
                }
            }
            idle_t0 = 0;
            if ((long long)e >= 0) {
                const int row = (int)(e & 0x0FFFFFFFu), mode = (int)((e >> 28) & 3u);
                item = make_int4(row, (int)tile, entry_gj(e), mode);
                // the group's next row becomes this producer's read-ahead candidate
                // (read-ahead entries carry no kEntryNext: one row ahead at most)
                if (p.read_ahead && (e & kEntryNext)) ra_e = queue_entry(entry_gj(e) + 1, row + 1, mode);
            }
        }
        if (timed_out) atomicOr(p.status, kStatusTimeout);
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
        if (p.host_logits) {
            // logits in mapped host memory: the compute warps copy the tile
            // themselves (host_tile_copy); the item is posted now
            mbar_arrive(&sm.full[stage]);
        } else {
            mbar_arrive_expect_tx(&sm.full[stage], bytes);
            bulk_load(stages + (size_t)stage * kTileBytes, src, bytes, &sm.full[stage],
                      item.w == kModeNatural ? npolicy : policy);
        }
        trace(p, kTrIssue, item.x, item.y, true);
        if (++stage == S) {
            stage = 0;
            phase ^= 1u;
        }
        // the next chained claim, and the next fresh item with its entry (depth-0
        // entries are all published), overlapping the next stage wait
        if (chain_claim == kNone && !chains_over) claim_chain();
        if (!fresh_done && fresh_ahead == kNone) {
            fresh_ahead = atomicAdd(&ctrl->fresh_next, 1u);
            fresh_done = fresh_ahead >= fresh_items;
            if (!fresh_done) fresh_entry = vload(&p.queue[fresh_ahead / T]);
        }
    }
}

// ------------------------------------------------------------------ tile: natural-alternative summary
//
// A natural-alternative tile keeps no candidates.  Each compute warp writes the
// four largest maxima of its 32 threads (each thread's maximum over its 8
// vectors, from pass 1) with their positions: summary entry
//   (ord32(thread maximum) << 32) | (tile << 8) | thread,   0 = none
// (threads whose lanes all lie past V have none).  The record stage turns the
// row's entries into a threshold theta below which no natural alternative can
// lie, and re-reads only the threads whose maximum reaches it (natural_record).


// The warp's four largest thread maxima u (ord32, 0 = none), largest first:
// lane r < 4 receives entry r.  Equal maxima are taken lowest lane first.
__device__ __forceinline__ unsigned long long warp_summary(uint32_t u, int lane, uint32_t pos_base) {
    unsigned long long mine = 0ull;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const uint32_t v = __reduce_max_sync(kFull, u);
        const unsigned b = __ballot_sync(kFull, u == v);
        const int l = __ffs(b) - 1;
        if (lane == r && v != 0u) mine = ((unsigned long long)v << 32) | (unsigned long long)(pos_base + (uint32_t)l);
        if (lane == l) u = 0u;
    }
    return mine;
}

// Tile element id (within the tile) of the thread's first element equal to m,
// from the vector maxima: the first vector whose maximum equals m, then the
// first element of that vector equal to m.
template <int ELT, bool FULL>
__device__ __forceinline__ int first_equal(const unsigned char* sp, int tid, int nv, float m,
                                           const uint32_t (&cm)[TileLayout<ELT>::NCH]) {
    using L = TileLayout<ELT>;
    int cf = L::NCH - 1;
#pragma unroll
    for (int c = L::NCH - 1; c >= 0; --c) cf = (vec_max<ELT>(cm[c]) == m) ? c : cf;
    const uint4 v = ld_vec<ELT, FULL>(sp, cf, tid, nv);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    int ef = L::EPV - 1;
#pragma unroll
    for (int e = L::EPV - 1; e >= 0; --e) {
        const float x = (ELT == 2) ? ((e & 1) ? bf16_hi(w[e >> 1]) : bf16_lo(w[e >> 1])) : __uint_as_float(w[e]);
        ef = (x == m) ? e : ef;
    }
    return (cf * kConsumerThreads + tid) * L::EPV + ef;
}

// The best 32 of two descending lists (one key per lane), descending.
template <typename T>
__device__ __forceinline__ T merge_lists(T a, T b, int lane) {
    const T rev = __shfl_sync(kFull, b, 31 - lane);
    return warp_bitonic_clean_desc(rev > a ? rev : a, lane);
}

__device__ __noinline__ bool decide_row(const Params& p, int2* cur, uint32_t ep);

// The compute warp's share of one tile: passes, the summary of its thread
// maxima (natural tiles), its partial results published to global memory
// ((max, exp-sum) and the argmax key, atomicMax on the row's best key), then
// the tile handed to the helper warp through a done slot.  The warps of a CTA
// never wait for one another.  FULL = false for the last, partial tile of a
// row (its lanes past V already -inf in the stage).  SCORE: prompt scoring
// (the count of logits above the target's is kept too; a separate instance,
// so generation runs carry none of it).  False after a timeout.
template <int ELT, bool FULL, bool SCORE>
__device__ __forceinline__ bool tile_work(const Params& p, Shared& sm, const unsigned char* sp, int nv, int tbase,
                                          const int4& info, int stage, int& ds, uint32_t& dphase,
                                          unsigned long long deadline, uint32_t ep) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int mode = info.w;
    const bool natural = mode == kModeNatural;
    const long long tslot = (long long)info.x * p.T + info.y;
    // prompt scoring: the target's logit, loaded now and used after pass 1
    float xt = 0.0f;
    if (SCORE && lane == 0) xt = load_logit<ELT>(p, info.x, __ldg(&p.targets[info.x]));
    // pass 1: maxima (per vector for a full tile)
    uint32_t cm[TileLayout<ELT>::NCH];
    const float m = stage_max<ELT, FULL>(sp, tid, nv, cm);
    const uint32_t om = ord32(__fadd_rn(m, 0.0f));
    const uint32_t omx = __reduce_max_sync(kFull, om);
    // argmax key: smallest id among the lanes holding the warp maximum
    uint32_t id = 0xFFFFFFFFu;
    if (om == omx && m > kNegInf) id = (uint32_t)(tbase + first_equal<ELT, FULL>(sp, tid, nv, m, cm));
    const uint32_t idmin = __reduce_min_sync(kFull, id);
    const unsigned long long wkey = ((unsigned long long)omx << 32) | (unsigned long long)(~idmin);
    // into the row's best key now; its result is waited for before the tile is
    // handed over (below), long after it returned
    unsigned long long prev_best = 0ull;
    if (lane == 0) prev_best = atomicMax(&p.row_best[info.x], wkey);
    // Partials that the record kernel reads are published with atomic
    // exchanges issued here and waited for before the tile is handed over
    // (below), so they are performed at their point of coherence before the
    // tile is counted, like the best key; their latency overlaps pass 2.  (The
    // (max, exp-sum) pair, known only after pass 2, is run-tagged instead.)
    unsigned long long prev_pub = 0ull;
    if (natural) {
        // the warp's four largest thread maxima, with their positions
        const unsigned long long e =
            warp_summary(m > kNegInf ? om : 0u, lane, ((uint32_t)info.y << 8) | (uint32_t)(warp * 32));
        if (lane < 4) prev_pub = atomicExch(&p.part_keys[tslot * kKeysPerTile + warp * 4 + lane], e);
    }
    if constexpr (SCORE) {
        if (natural) {
            // prompt scoring: this warp's lanes whose logit is above the target's,
            // and the smallest of those logits (the rank is finished in the record
            // kernel, once lse is known); vectors whose maximum is not above it
            // are skipped
            const float t = __shfl_sync(kFull, xt, 0);
            int cnt = 0;
            float mn = kPosInf;
#pragma unroll
            for (int c = 0; c < TileLayout<ELT>::NCH; ++c) {
                if (!(vec_max<ELT>(cm[c]) > t)) continue;
                const uint4 v = ld_vec<ELT, FULL>(sp, c, tid, nv);
                const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < TileLayout<ELT>::EPV; ++e) {
                    const float x = (ELT == 2) ? ((e & 1) ? bf16_hi(w4[e >> 1]) : bf16_lo(w4[e >> 1]))
                                               : __uint_as_float(w4[e]);
                    if (x > t) {
                        ++cnt;
                        mn = fminf(mn, x);
                    }
                }
            }
            cnt = (int)__reduce_add_sync(kFull, (unsigned)cnt);
            mn = warp_min_f(mn);
            if (lane == 4)
                prev_pub = atomicExch(reinterpret_cast<unsigned long long*>(&p.part_rank[tslot * kWarps + warp]),
                                      ((unsigned long long)__float_as_uint(mn) << 32) | (uint32_t)cnt);
        }
    }
    // pass 2: sum exp(x - m) = 2^(x*log2e - mb - mb_lo): mb_lo, the rounding
    // residual of m*log2e, is applied once, so large |m| costs no accuracy
    float s = 0.0f;
    if (mode != kModeArgmax && m > kNegInf) {
        const float mb = m * kLog2e;
        const float mb_lo = fmaf(m, kLog2e, -mb);
        s = stage_expsum<ELT, FULL>(sp, tid, nv, mb) * ex2(-mb_lo);
    }
    // partial results of the warp, then the tile goes to the helper warp
    // through a done slot: once the 8 warps arrived, it counts the tile for
    // the row
    if (!FULL) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the -inf fill, before the next copy
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[stage]);  // no more reads of this stage by this warp
    const float Mw = unord32(omx);
    const float sc = (m > kNegInf && mode != kModeArgmax) ? s * ex2((m - Mw) * kLog2e) : 0.0f;
    const float sw = warp_sum_f(sc);
    if (lane == 0)
        st_tagged(&p.part_ms[tslot * kWarps + warp], tagged(ep, __float_as_uint(Mw)), tagged(ep, __float_as_uint(sw)));
    // every lane's exchange result, gathered (a warp-wide reduction waits for all of them)
    const uint32_t pub = __reduce_or_sync(kFull, (uint32_t)prev_pub ^ (uint32_t)(prev_pub >> 32));
    if (__any_sync(kFull, !mbar_wait(&sm.dfree[ds], (dphase >> ds) & 1u, deadline))) {  // slot read
        if (lane == 0) atomicOr(p.status, kStatusTimeout);
        return false;
    }
    if (lane == 0) {
        if (warp == 0) sm.dslot[ds] = make_int4(info.x, info.z, 0, 0);
        // the best-key update and the exchanges must have returned (so they are
        // performed at their point of coherence) before the count that follows
        // the arrival: the store of their results cannot issue before the
        // results are back
        sm.wbest[warp] = prev_best ^ pub;
        mbar_arrive(&sm.dfull[ds]);
    }
    dphase ^= 1u << ds;
    if (++ds == kDoneRing) ds = 0;
    return true;
}

// ------------------------------------------------------------------ compute warps
//
// Each compute warp reduces its share of every tile on its own and publishes
// its partial results itself: the warps never wait for one another, except on
// natural-alternative tiles, where the 8 warp thresholds and candidates are
// exchanged through a candidate slot (bounded mbarrier waits).
// Logits in pinned host memory mapped into the device's address space (TMA
// bulk copies are kept for device memory): each compute thread copies its own
// 16-byte vectors of the tile, the only ones it reads, so a warp moves 512
// contiguous bytes per instruction and no block barrier is needed before the
// reads.
template <int ELT>
__device__ __noinline__ void host_tile_copy(const Params& p, unsigned char* sp, int row, int tbase, int nv) {
    const int tid = threadIdx.x;
    const uint32_t bytes = (static_cast<uint32_t>(nv * ELT) + 15u) & ~15u;
    const unsigned char* src = reinterpret_cast<const unsigned char*>(p.logits) + ((long long)row * p.Vp + tbase) * ELT;
#pragma unroll
    for (int c = 0; c < TileLayout<ELT>::NCH; ++c) {
        const uint32_t o = static_cast<uint32_t>(c * kConsumerThreads + tid) * 16u;
        if (o < bytes)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(sp + o)), "l"(src + o) : "memory");
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
}

template <int ELT, bool SCORE>
__device__ void compute_loop(const Params& p, Shared& sm, unsigned char* stages, unsigned long long t0, uint32_t ep) {
    constexpr int S = StageCfg<ELT>::kStages;
    constexpr int kTE = tile_elems<ELT>();
    const int tid = threadIdx.x, lane = tid & 31;
    const unsigned long long deadline = t0 + p.timeout_ns;
    const int V = (int)p.V;
    int stage = 0, ds = 0;
    uint32_t phase = 0;
    uint32_t dphase = 0;              // dphase bit r: uses of done slot r, mod 2
    for (;;) {
        if (__any_sync(kFull, !mbar_wait(&sm.full[stage], phase, deadline))) {
            if (lane == 0) atomicOr(p.status, kStatusTimeout);
            return;
        }
        const int4 info = sm.info[stage];
        if (info.z < 0) return;  // no more tiles
        const unsigned char* sp = stages + (size_t)stage * kTileBytes;
        const int tile = info.y;
        const int tbase = tile * kTE;
        const int rem = V - tbase;
        const int nv = rem < kTE ? (rem > 0 ? rem : 0) : kTE;
        if (p.host_logits) host_tile_copy<ELT>(p, stages + (size_t)stage * kTileBytes, info.x, tbase, nv);
        trace(p, kTrTileStart, info.x, tile, tid == 0);
        bool ok;
        if (__builtin_expect(nv == kTE, 1)) {
            ok = tile_work<ELT, true, SCORE>(p, sm, sp, nv, tbase, info, stage, ds, dphase, deadline, ep);
        } else {
            fill_partial<ELT>(stages + (size_t)stage * kTileBytes, tid, nv);
            ok = tile_work<ELT, false, SCORE>(p, sm, sp, nv, tbase, info, stage, ds, dphase, deadline, ep);
        }
        if (!ok) return;
        trace(p, kTrTileEnd, info.x, tile, tid == 0);
        if (++stage == S) {
            stage = 0;
            phase ^= 1u;
        }
    }
}

// ------------------------------------------------------------------ decisions

// Acceptance decision of the row *cur = (row, queue entry), whose tiles are
// all counted and whose parent accepted (lane 0 of the compute warp whose
// increment completed it): argmax = the row's best key.  On acceptance the
// next row of the group must be read: its queue entry is appended (flagged
// when read-ahead has already claimed some or all of its tiles), it is marked
// for decision, and the row after it becomes a read-ahead candidate.
// Otherwise the group ends and read-ahead on the next row stops.  A
// requesting row is flagged for the record kernel.  Returns true, with *cur
// advanced to the next row, when read-ahead had already counted every tile of
// that row: the caller decides it too.
__device__ __noinline__ bool decide_row(const Params& p, int2* cur, uint32_t ep) {
    const unsigned T = (unsigned)p.T;
    const unsigned fresh_rows = vload(&p.ctrl->fresh_rows);
    const int row = cur->x, entry = cur->y;
    const int g = entry >> 4, j = entry & 15;
    const int4 d = __ldcg(&p.gdesc[g]);
    const unsigned long long bk = atomicMax(&p.row_best[row], 0ull);  // read at its point of coherence
    const int draft = p.drafts != nullptr ? __ldg(&p.drafts[row]) : -1;  // none when scoring
    const int eos = p.eos != nullptr ? __ldg(&p.eos[g]) : -1;
    const int r0 = d.x, k = d.y & 0xFF, req = (d.y >> 13) & 1, samp = d.w, mode = (d.y >> 8) & 3;
    const uint32_t amax = key_id(bk);
    const int chosen = (k == 0 && samp >= 0) ? samp : (int)amax;
    // commit clipping: an emitted EOS token ends the group (it stays emitted)
    const bool accept = (j < k) && (draft == (int)amax) && !(eos >= 0 && chosen == eos);
    int next_done = 0;
    if (accept) {
        // independent round trips, issued together
        const unsigned pos = fresh_rows + atomicAdd(&p.ctrl->chain_tail, 1u);
        unsigned long long e = queue_entry((g << 4) | (j + 1), row + 1, mode);
        if (p.read_ahead) {
            const unsigned claimed = atomicCAS(&p.tclaim[row + 1], 0u, kClosed);
            next_done = atomicAdd(&p.done[row + 1], kParentDone);
            if (j + 2 <= k) e |= kEntryNext;
            if (claimed != 0u) e |= claimed >= T ? kEntrySkip : kEntryShared;
        }
        vstore(&p.queue[pos], e);
    } else if (p.read_ahead && j < k) {
        atomicAdd(&p.tclaim[row + 1], kClosed);  // the next row is not needed
    }
    if (p.emitted != nullptr) {  // generation outputs (none when scoring)
        p.emitted[row] = chosen;
        if (!accept) {
            p.accepted[g] = j;
            for (int jj = j + 1; jj <= k; ++jj) p.emitted[r0 + jj] = -1;
        }
    }
    if (req) {  // a record task for the record kernel (or the sharded kernels)
        if (chosen >= p.V) atomicOr(p.status, kStatusBadToken);
        const unsigned i = atomicAdd(&p.ctrl->rec_count, 1u);
        const int is_amax = (k == 0 && samp >= 0) ? 0 : 1;  // the chosen logit is then the row maximum
        const uint32_t dw = (uint32_t)((d.y & 0x3FFF) | (is_amax << 14) | (d.z << 16));
        st_tagged(&p.rec_tasks[2 * (size_t)i], tagged(ep, (uint32_t)chosen), tagged(ep, (uint32_t)row));
        st_tagged(&p.rec_tasks[2 * (size_t)i + 1], tagged(ep, dw), tagged(ep, (uint32_t)g));
    }
    trace(p, kTrDecision, row, accept ? 1 : 0, true);
    if (!accept) {
        // the record flag and the emitted tokens are written before the group retires
        atomicSub(&p.ctrl->outstanding, 1);
        return false;
    }
    *cur = make_int2(row + 1, entry + 1);
    return next_done == (int)T;  // else decided by the increment that completes it
}

// ------------------------------------------------------------------ helper warp
//
// Takes the compute warps' tiles through the done slots, in order: counts each
// tile for its row and decides the row when its increment completes it.  The
// compute warps never wait on a count or a decision.  Stops when every compute
// warp has finished and the next slot holds nothing.
//
// Ordering without fences.  A decision needs the row's best key complete:
// every compute warp waits for the result of its best-key atomicMax before
// its done-slot arrival, so the update has been performed at the key's
// point of coherence (the L2 slice that owns it) before the count is issued,
// and the decider reads the key with an atomic at that same point after its
// own count returned.  The record kernel reads the tile partials and record
// tasks while this grid runs: they are run-tagged, or were performed before
// their tiles were counted (see tile_work).  (An acquire-
// release count gives the same order through the memory model, but its fence
// waits for the multiprocessor's outstanding memory traffic, which made the
// helper's per-tile counts the bottleneck.)
template <int ELT>
__device__ __noinline__ void helper_loop(const Params& p, Shared& sm, unsigned long long deadline, uint32_t ep) {
    const int lane = threadIdx.x & 31;
    int ds = 0;
    uint32_t dphase = 0;
    for (uint32_t i = 0;; ++i) {
        // polled (this warp has nothing else to wait on); lane 0's view decides for the warp
        if (__shfl_sync(kFull, (int)mbar_test_wait(&sm.dfull[ds], (dphase >> ds) & 1u), 0)) {
            const int4 d = sm.dslot[ds];
            __syncwarp();
            int old = 0;
            if (lane == 0) {
                mbar_arrive(&sm.dfree[ds]);  // the slot's contents are read
                old = atomicAdd(&p.done[d.x], 1);
            }
            dphase ^= 1u << ds;
            if (++ds == kDoneRing) ds = 0;
            if (lane == 0 && old == p.done_last) {
                int2 cur = make_int2(d.x, d.y);
                while (decide_row(p, &cur, ep)) {
                }
            }
            __syncwarp();
            continue;
        }
        if (vload(&sm.sel_exit) == kWarps) {
            __threadfence_block();  // every arrival precedes the last exit count
            if (!__any_sync(kFull, mbar_test_wait(&sm.dfull[ds], (dphase >> ds) & 1u))) return;
            continue;
        }
        if ((i & 63u) == 63u && globaltimer() > deadline) {
            if (lane == 0) atomicOr(p.status, kStatusTimeout);
            return;
        }
    }
}

template <int ELT, bool SCORE>
__global__ void __launch_bounds__(kThreads, StageCfg<ELT>::kMinBlocks) lp_stream_kernel(Params p) {
    constexpr int S = StageCfg<ELT>::kStages;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    // the stages start on a 128-byte boundary (the static event counters come
    // first).  At a 16-byte offset, every 32-byte sector of the 16-byte
    // per-thread copies was fetched twice, and the bulk copies ran slower.
    unsigned char* stages = smem_raw + ((kStageAlign - (smem_u32(smem_raw) & (kStageAlign - 1u))) & (kStageAlign - 1u));
    Shared& sm = *reinterpret_cast<Shared*>(stages + (size_t)S * kTileBytes);
    const int tid = threadIdx.x;
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kWarps);
        }
        g_trace_n[0] = g_trace_n[1] = g_trace_n[2] = 0u;
        for (int s = 0; s < kDoneRing; ++s) {
            mbar_init(&sm.dfull[s], kWarps);
            mbar_init(&sm.dfree[s], 1);
            mbar_arrive(&sm.dfree[s]);  // the slot starts free (its phase 0 is complete)
        }
        sm.sel_exit = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    // While the prepare kernel runs, each CTA brings into L2 the tiles of the
    // first claims it stands for: ticket blockIdx.x + w * gridDim.x (w <
    // LP_EARLY_PREFETCH), tile ticket % T of queue position ticket / T, taken
    // to be group ticket / T's first row (every group read).  The inputs are
    // the caller's, complete before the prepare kernel started; a guess that
    // misses only costs its read.
    if (LP_EARLY_PREFETCH > 0 && tid == kConsumerThreads && !p.host_logits) {
        const long long T = p.T;
        const long long row_bytes = ((long long)p.V * ELT + 15) & ~15ll;
        for (int w = 0; w < LP_EARLY_PREFETCH; ++w) {
            const long long t = (long long)blockIdx.x + (long long)w * gridDim.x;
            const long long q = t / T;
            if (q >= p.G) break;
            const int row = p.targets != nullptr ? (int)q : __ldg(&p.indptr[q]);
            if (row < 0 || row >= p.rows) continue;
            const long long off = (t % T) * (long long)kTileBytes;
            if (off >= row_bytes) continue;
            const uint32_t sz = (uint32_t)min((long long)kTileBytes, row_bytes - off);
            const unsigned char* a = reinterpret_cast<const unsigned char*>(p.logits) + (long long)row * p.Vp * ELT + off;
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a), "r"(sz) : "memory");
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // the record kernel may be scheduled now (the prepare kernel's writes are
    // visible): its CTAs take the multiprocessor room this grid leaves, and
    // more as its CTAs exit, and build each record as its task appears
    asm volatile("griddepcontrol.launch_dependents;");
    if (vload(&p.ctrl->abort) != 0u) return;
    const uint32_t ep = vload(&p.ctrl->epoch);
    const unsigned long long t0 = globaltimer();
    trace(p, kTrKernel, 0, 0, tid == 0);
    const int warp = tid >> 5;
    if (warp == kWarps) {
        const FirstClaim first = first_claim(p);
        if (tid == kConsumerThreads) producer_loop<ELT>(p, sm, stages, t0, first);
        return;
    }
    if (warp == kWarps + 1) {
        helper_loop<ELT>(p, sm, t0 + p.timeout_ns, ep);
        return;
    }
    compute_loop<ELT, SCORE>(p, sm, stages, t0, ep);
    if ((tid & 31) == 0) {
        __threadfence_block();  // this warp's slot arrivals come first
        atomicAdd(&sm.sel_exit, 1);
    }
}

// ------------------------------------------------------------------ records

// ---- natural alternatives of a record (one CTA of 256 threads, the 8 compute warps)
//
// The row's summary entries (each compute warp's 4 largest thread maxima, per
// natural tile) give a threshold theta such that at least 32 entries, so 32
// distinct lanes, are >= theta: warp w of the record CTA takes the entries of
// warp column w of every tile and finds their 4th largest; theta is the
// smallest of the 8.  Every lane >= theta lies in a thread whose maximum
// reaches theta.  Such a thread is either named by an entry >= theta, or it is
// not among its warp share's 4 largest, and then the share's 4th entry reaches
// theta too: that share is re-read whole.  So C = {v : x_v >= theta} is
// gathered exactly, from a few threads' vectors.  C holds the row's 32 largest
// logits, and fl32(x - lse) is non-decreasing in x, so every lane outside C has
// a logprob <= lp(x') for the largest float x' below theta: if that is below
// the K-th logprob L of C, the K best of C by (logprob desc, id asc) are the
// row's; otherwise the lanes equal to L are collected over the whole row in id
// order (subtraction ties across theta, rare).  A row whose entries cannot
// give a theta (a tiny vocabulary) takes every lane; a row whose candidates
// overflow the shared-memory lists (long runs of equal values) takes the exact
// path of natural_exact.

// Element e (0..EPV-1) of a 16-byte vector.
template <int ELT>
__device__ __forceinline__ float vec_elem(const uint4& v, int e) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    if constexpr (ELT == 2) return (e & 1) ? bf16_hi(w[e >> 1]) : bf16_lo(w[e >> 1]);
    else return __uint_as_float(w[e]);
}

// Logprob key: descending order = (lp desc, id asc).
__device__ __forceinline__ unsigned long long lp_key(float x, float lse, uint32_t id) {
    return (static_cast<unsigned long long>(ord32(logprob(x, lse))) << 32) | static_cast<unsigned long long>(~id);
}

// The part of a row a natural selection covers: tiles [t0, t1), ids [v0, v1)
// (the whole row, or one vocabulary shard of whole tiles).
struct Span {
    int t0, t1;
    long long v0, v1;
};

// Warp 0 writes, from pair slot `from` on, the lanes of the span whose
// logprob equals L, smallest ids first, until keff pairs are written.
template <int ELT>
__device__ __forceinline__ void fill_equal_lanes(const Params& p, int* rec, int row, const Span& sp, float lse, float L,
                                                 int from, int keff, int lane) {
    const unsigned lbits = __float_as_uint(L);
    int got = from;
    for (long long v0 = sp.v0; v0 < sp.v1 && got < keff; v0 += 32) {
        const long long v = v0 + lane;
        const bool m = v < sp.v1 && logprob(load_logit<ELT>(p, row, v), lse) == L;
        const unsigned bb = __ballot_sync(kFull, m);
        const int before = __popc(bb & ((1u << lane) - 1u));
        if (m && got + before < keff) {
            rec[2 + 2 * (got + before)] = (int)v;
            rec[3 + 2 * (got + before)] = (int)lbits;
        }
        got += __popc(bb);
    }
}

// The natural pairs of the record (into sm.rec), exact but slow: for rows
// whose candidates overflow the lists.  L = the K-th largest logprob, found as
// lp of the K-th largest logit (bisection over the ordered bit patterns of the
// logits, each step a count over the row); then the lanes above L (fewer than
// K, sorted by one warp) and the smallest ids equal to L.
template <int ELT>
__device__ __noinline__ void natural_exact(const Params& p, RecShared& sm, int row, const Span& sp, int keff, float lse) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // the largest o with count(ord32(x) >= o) >= keff
    uint32_t lo = ord32(kNegInf), hi = ord32(kPosInf);
    while (lo < hi) {
        const uint32_t mid = lo + ((hi - lo + 1u) >> 1);
        int c = 0;
        for (long long v = sp.v0 + tid; v < sp.v1; v += kConsumerThreads)
            c += ord32(__fadd_rn(load_logit<ELT>(p, row, v), 0.0f)) >= mid;
        c = (int)__reduce_add_sync(kFull, (unsigned)c);
        if (lane == 0) sm.red_x[warp] = c;
        cbar();
        int tot = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) tot += sm.red_x[w];
        cbar();
        if (tot >= keff) lo = mid;
        else hi = mid - 1u;
    }
    const float L = logprob(unord32(lo), lse);
    // lanes reported above L: fewer than keff
    if (tid == 0) sm.n_keys = 0;
    cbar();
    for (long long v = sp.v0 + tid; v < sp.v1; v += kConsumerThreads) {
        const float x = load_logit<ELT>(p, row, v);
        if (logprob(x, lse) > L) {
            const int i = atomicAdd(&sm.n_keys, 1);
            if (i < 32) sm.ckeys[i] = lp_key(x, lse, (uint32_t)v);
        }
    }
    cbar();
    if (warp == 0) {
        const int c_gt = sm.n_keys < 32 ? sm.n_keys : 32;
        const unsigned long long k = warp_sort_desc(lane < c_gt ? sm.ckeys[lane] : 0ull, lane);
        if (lane < c_gt) {
            sm.rec[2 + 2 * lane] = (int)key_id(k);
            sm.rec[3 + 2 * lane] = (int)__float_as_uint(key_value(k));
        }
        fill_equal_lanes<ELT>(p, sm.rec, row, sp, lse, L, c_gt, keff, lane);
    }
    cbar();
}

// The record's fast path keeps up to kCachedShares warp shares per thread in
// registers (rows of up to 32 * kCachedShares tiles).
constexpr int kCachedShares = 2;

// Step 1 (before the record's first barrier): thread (w, lane) takes the
// shares of warp column w in tiles lane, lane + 32, ...; the warp's 8 largest
// entry values go to sm.wtop[w] (0: none).  The 32nd largest of those 64
// values is a threshold with at least 32 entries at or above it.
constexpr int kWarpTop = 8;
__device__ __forceinline__ void summary_top(const Params& p, RecShared& sm, long long base, const Span& sp, int warp,
                                            int lane) {
    uint32_t top[4] = {0u, 0u, 0u, 0u};  // this thread's 4 largest entry values, descending
    for (int t = sp.t0 + lane; t < sp.t1; t += 32) {
        const ulonglong2* q = reinterpret_cast<const ulonglong2*>(p.part_keys + (base + t) * kKeysPerTile + warp * 4);
        const ulonglong2 a = __ldcg(q), b = __ldcg(q + 1);
        const unsigned long long e[4] = {a.x, a.y, b.x, b.y};
#pragma unroll
        for (int r = 0; r < 4; ++r) {  // insert
            uint32_t v = (uint32_t)(e[r] >> 32);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t hi = v > top[k] ? v : top[k], lo = v > top[k] ? top[k] : v;
                top[k] = hi;
                v = lo;
            }
        }
    }
    // the warp's 8 largest: knock out the largest head eight times.  A thread
    // keeps only its own 4 largest; if it held more of the warp's 8, smaller
    // values are taken instead, still each the value of a distinct entry, so
    // the count behind the threshold holds.
#pragma unroll
    for (int r = 0; r < kWarpTop; ++r) {
        const uint32_t v = __reduce_max_sync(kFull, top[0]);
        const unsigned b = __ballot_sync(kFull, top[0] == v);
        if (lane == __ffs(b) - 1) {
            top[0] = top[1];
            top[1] = top[2];
            top[2] = top[3];
            top[3] = 0u;
        }
        if (lane == r) sm.wtop[warp][r] = v;
    }
}

// Steps 4-5 of a natural selection, once sm.ckeys[0, sm.n_keys) holds the
// logprob keys of every lane >= theta (sm.theta_o, 0: every lane of the span)
// and the block has synchronised: the best keff keys by rank into the record's
// pairs, then the subtraction-tie check across theta.
template <int ELT>
__device__ __noinline__ void natural_rank(const Params& p, RecShared& sm, int row, const Span& sp, int keff, float lse) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t th = sm.theta_o;
    const float theta = th ? unord32(th) : kNegInf;
    if (sm.n_keys > kCandKeys) {
        natural_exact<ELT>(p, sm, row, sp, keff, lse);
        return;
    }
    // 4. the best keff keys by rank (keys are distinct: they carry the id)
    const int nk = sm.n_keys;
    for (int j = nk + tid; j < ((nk + 7) & ~7); j += kConsumerThreads) sm.ckeys[j] = 0ull;  // pad to 8
    cbar();
    for (int i = tid; i < nk; i += kConsumerThreads) {
        const unsigned long long k = sm.ckeys[i];
        int r0 = 0, r1 = 0, r2 = 0, r3 = 0;
        for (int j = 0; j < nk; j += 8) {
            const ulonglong2 a = *reinterpret_cast<const ulonglong2*>(&sm.ckeys[j]);
            const ulonglong2 b = *reinterpret_cast<const ulonglong2*>(&sm.ckeys[j + 2]);
            const ulonglong2 c = *reinterpret_cast<const ulonglong2*>(&sm.ckeys[j + 4]);
            const ulonglong2 d = *reinterpret_cast<const ulonglong2*>(&sm.ckeys[j + 6]);
            r0 += (a.x > k) + (a.y > k);
            r1 += (b.x > k) + (b.y > k);
            r2 += (c.x > k) + (c.y > k);
            r3 += (d.x > k) + (d.y > k);
        }
        const int rank = r0 + r1 + r2 + r3;
        if (rank < keff) {
            sm.rec[2 + 2 * rank] = (int)key_id(k);
            sm.rec[3 + 2 * rank] = (int)__float_as_uint(key_value(k));
            if (rank == keff - 1) sm.lkey = k;
        }
    }
    cbar();
    // 5. lanes below theta can tie with the K-th logprob only if the float just
    // below theta already reports it
    const float L = key_value(sm.lkey);
    if (th != 0u && logprob(nextafterf(theta, kNegInf), lse) == L) {
        if (tid == 0) sm.n_thr = 0;
        cbar();
        int gt = 0;
        for (int i = tid; i < nk; i += kConsumerThreads) gt += key_value(sm.ckeys[i]) > L;
        gt = (int)__reduce_add_sync(kFull, (unsigned)gt);
        if (lane == 0 && gt) atomicAdd(&sm.n_thr, gt);
        cbar();
        if (warp == 0) fill_equal_lanes<ELT>(p, sm.rec, row, sp, lse, L, sm.n_thr, keff, lane);
        cbar();
    }
}

// Steps 2-5, all 256 threads, after warp 0 has set sm.theta_o (0: every lane
// is a candidate) and sm.lse: candidates, their logprob keys, the best keff by
// rank, the subtraction-tie check.  Writes the natural pairs into sm.rec.
template <int ELT>
__device__ __noinline__ void natural_record(const Params& p, RecShared& sm, int row, long long base, const Span& sp,
                                            int keff) {
    constexpr int TE = tile_elems<ELT>(), EPV = 16 / ELT, NCH = TileLayout<ELT>::NCH;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float lse = sm.lse;
    const uint32_t th = sm.theta_o;
    const float theta = th ? unord32(th) : kNegInf;
    const long long V = sp.v1;  // lanes at or past it are not the span's
    const unsigned char* rowp = reinterpret_cast<const unsigned char*>(p.logits) + (long long)row * p.Vp * ELT;
    bool overflow = false;
    if (th == 0u) {
        // no threshold (a tiny vocabulary): every lane is a candidate
        const long long n = sp.v1 - sp.v0;
        if (n > kCandKeys) {
            overflow = true;
        } else {
            for (int i = tid; i < n; i += kConsumerThreads)
                sm.ckeys[i] = lp_key(load_logit<ELT>(p, row, sp.v0 + i), lse, (uint32_t)(sp.v0 + i));
            if (tid == 0) sm.n_keys = (int)n;
        }
        cbar();
    } else {
        // 2. candidate threads: entries >= theta, and whole shares whose 4th entry reaches it
        int i = 0;
        for (int t = sp.t0 + lane; t < sp.t1; t += 32, ++i) {
            unsigned long long e[4];
            {
                const ulonglong2* q = reinterpret_cast<const ulonglong2*>(p.part_keys + (base + t) * kKeysPerTile + warp * 4);
                const ulonglong2 a = __ldcg(q), b = __ldcg(q + 1);
                e[0] = a.x; e[1] = a.y; e[2] = b.x; e[3] = b.y;
            }
            if (e[3] != 0ull && (uint32_t)(e[3] >> 32) >= th) {
                const int k = atomicAdd(&sm.n_sh, 1);
                if (k < kCandShares) sm.csh[k] = (uint32_t)(t * kWarps + warp);
            } else {
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    if (e[r] != 0ull && (uint32_t)(e[r] >> 32) >= th) {
                        const int k = atomicAdd(&sm.n_thr, 1);
                        if (k < kCandThreads) sm.cthr[k] = (uint32_t)e[r];
                    }
                }
            }
        }
        cbar();
        const int nthr = sm.n_thr, nsh = sm.n_sh;
        overflow = nthr > kCandThreads || nsh > kCandShares;
        if (!overflow) {
            // 3. their vectors, re-read from global memory (4 loads in flight per
            // thread): keys of the lanes >= theta
            const int items = (nthr + nsh * 32) * NCH;
            for (int it0 = 0; it0 < items; it0 += 4 * kConsumerThreads) {
                uint4 x[4];
                long long v0[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int it = it0 + u * kConsumerThreads + tid;
                    v0[u] = V;
                    if (it < items) {
                        const int c = it % NCH, j = it / NCH;
                        uint32_t pos;  // tile << 8 | thread
                        if (j < nthr) {
                            pos = sm.cthr[j];
                        } else {
                            const uint32_t sh = sm.csh[(j - nthr) >> 5];
                            pos = ((sh / kWarps) << 8) | ((sh % kWarps) * 32u + (uint32_t)((j - nthr) & 31));
                        }
                        v0[u] = (long long)(pos >> 8) * TE + (long long)(c * kConsumerThreads + (int)(pos & 0xFFu)) * EPV;
                    }
                    if (v0[u] < V) x[u] = __ldcs(reinterpret_cast<const uint4*>(rowp + v0[u] * ELT));
                }
                // warp-aggregated appends: one shared atomic per warp and round
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    int n = 0;
                    if (v0[u] < V) {
#pragma unroll
                        for (int e = 0; e < EPV; ++e) n += (v0[u] + e < V && vec_elem<ELT>(x[u], e) >= theta) ? 1 : 0;
                    }
                    if (!__any_sync(kFull, n > 0)) continue;
                    int tot = n;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const int q = __shfl_up_sync(kFull, tot, o);
                        if (lane >= o) tot += q;
                    }
                    int k0 = 0;
                    if (lane == 31) k0 = atomicAdd(&sm.n_keys, tot);
                    int k = __shfl_sync(kFull, k0, 31) + tot - n;
                    if (n > 0) {
#pragma unroll
                        for (int e = 0; e < EPV; ++e) {
                            const float y = vec_elem<ELT>(x[u], e);
                            if (v0[u] + e < V && y >= theta) {
                                if (k < kCandKeys) sm.ckeys[k] = lp_key(y, lse, (uint32_t)(v0[u] + e));
                                ++k;
                            }
                        }
                    }
                }
            }
            cbar();
            overflow = sm.n_keys > kCandKeys;
        }
    }
    if (overflow) {
        natural_exact<ELT>(p, sm, row, sp, keff, lse);
        return;
    }
    natural_rank<ELT>(p, sm, row, sp, keff, lse);
}

// Prompt scoring: the largest float X with fl32(X - lse) <= lp, where lp =
// fl32(xt - lse) is the target's logprob.  x -> fl32(x - lse) is monotone, so a
// logit is reported strictly above the target exactly when it is above X, and
// the logits in (xt, X] are the ones whose logprob rounds to the target's.  A
// warp search over the ordered bit patterns in [xt, +inf]: each round the 32
// lanes test 32 points spread over the interval, and the interval shrinks to
// the gap between the last point that holds and the first that does not.
__device__ __forceinline__ float score_limit(float xt, float lse, float lp, int lane) {
    uint32_t lo = ord32(xt), hi = ord32(kPosInf);  // the predicate holds at lo
    if (__fsub_rn(kPosInf, lse) <= lp) return kPosInf;
    while (hi - lo > 1u) {
        const uint32_t q = lo + (uint32_t)(((unsigned long long)(hi - lo) * (unsigned)(lane + 1)) / 33ull);
        const bool ok = __fsub_rn(unord32(q), lse) <= lp;
        const int n = __popc(__ballot_sync(kFull, ok));  // the points that hold are a prefix
        const uint32_t nlo = __shfl_sync(kFull, q, n > 0 ? n - 1 : 0);
        const uint32_t nhi = __shfl_sync(kFull, q, n < 32 ? n : 31);
        lo = n > 0 ? nlo : lo;
        hi = n < 32 ? nhi : hi;
    }
    return unord32(lo);
}

// Merges two (max, sum exp(x - max)) pairs.
__device__ __forceinline__ void ms_merge(float& m, float& s, float m2, float s2) {
    const float M = fmaxf(m, m2);
    if (M == kNegInf) return;
    s = (m > kNegInf ? s * ex2((m - M) * kLog2e) : 0.0f) + (m2 > kNegInf ? s2 * ex2((m2 - M) * kLog2e) : 0.0f);
    m = M;
}

// A (max, exp-sum) tile partial of this run, by its words as loaded: it was
// written before its tile was counted, so it has landed or is about to; waits
// (bounded) until both words carry the run's epoch.
__device__ __noinline__ ulonglong2 part_ms_wait(const Params& p, long long i, ulonglong2 v, uint32_t ep,
                                                unsigned long long deadline) {
    while (!has_epoch(v, ep)) {
        if (globaltimer() > deadline) {
            atomicOr(p.status, kStatusTimeout);
            break;
        }
        v = ld_tagged(&p.part_ms[i]);
    }
    return v;
}

// Record of a requested, emitted row, built by one CTA of 256 threads.
//
// Every independent load is issued first (the tile partials, the summary
// entries, the chosen logit, the explicit ids; the explicit ids' logits as
// soon as the ids arrive).  Each warp then reduces its partials (maximum
// first, then the rescaled sums) and, for natural rows, finds the 8 largest
// summary entries of its warp column and starts loading those threads'
// vectors, so the candidate gather is in flight across the block barrier.
// After the barrier every warp derives the same lse and threshold theta from
// the warps' results (same operations in the same order, so the same bits),
// keeps the prefetched lanes >= theta as logprob keys and checks that its
// column has no candidate thread outside the 8 it loaded (no other entry >=
// theta, no warp share whose 4th entry reaches theta); if any warp finds one,
// the block takes the general path of natural_record.
// SCORE: the prompt-scoring record (rank, 43 words) instead of the 258-word one.
template <int ELT, bool SCORE>
__device__ __noinline__ void record_block(const Params& p, RecShared& sm, int row, int g, int chosen, int dy,
                                          int kc, uint32_t ep, unsigned long long deadline) {
    constexpr int TE = tile_elems<ELT>(), EPV = 16 / ELT;
    static_assert(TileLayout<ELT>::NCH == 8, "four lanes load a thread's 8 vectors, two each");
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int mode = (dy >> 8) & 3, ids = (dy >> 12) & 1;
    const bool chosen_is_max = ((dy >> 14) & 1) != 0;  // its logit is the row maximum
    const int T = p.T;
    const long long base = (long long)row * T;
    const bool natural = !ids && mode == kModeNatural && kc > 0;
    constexpr bool score = SCORE;
    const unsigned char* rowp = reinterpret_cast<const unsigned char*>(p.logits) + (long long)row * p.Vp * ELT;
    // ---- every independent load, issued together
    int id = -1;
    if (ids && tid < kc) id = __ldg(&p.token_ids[(long long)g * kMaxIds + tid]);
    float xc = 0.0f;
    if (tid == 32 && !chosen_is_max && chosen >= 0 && chosen < p.V) xc = load_logit<ELT>(p, row, chosen);
    const int np = T * kWarps;  // one (max, exp-sum) per warp of each tile
    ulonglong2 v[2];
#pragma unroll
    for (int u = 0; u < 2; ++u)
        if (tid + u * kConsumerThreads < np) v[u] = ld_tagged(&p.part_ms[base * kWarps + tid + u * kConsumerThreads]);
    // summary entries of warp column `warp`: tiles lane and lane + 32
    ulonglong2 ca[kCachedShares], cb[kCachedShares];
#pragma unroll
    for (int i = 0; i < kCachedShares; ++i) {
        const int t = lane + 32 * i;
        ca[i] = cb[i] = make_ulonglong2(0ull, 0ull);
        if (natural && t < T) {
            const ulonglong2* q = reinterpret_cast<const ulonglong2*>(p.part_keys + (base + t) * kKeysPerTile + warp * 4);
            ca[i] = __ldcg(q);
            cb[i] = __ldcg(q + 1);
        }
    }
    // the explicit ids' logits, once the ids are back
    float xi = 0.0f;
    if (ids && tid < kc && id >= 0 && id < p.V) xi = load_logit<ELT>(p, row, id);
    for (int w = tid; w < kRecordWords; w += kConsumerThreads)
        sm.rec[w] = (w >= 2 && (w & 1) == 0) ? -1 : (int)kUnusedBits;
    if (tid == 0) {
        sm.corr = 0;
        sm.n_thr = sm.n_sh = sm.n_keys = 0;
        sm.slow = 0;
    }
    // ---- (max, exp-sum) of the thread's partials, then of the warp's
    float m = kNegInf, s = 0.0f;
    int above = 0;  // prompt scoring: logits above the target's
    for (int t0 = tid; t0 < np; t0 += 2 * kConsumerThreads) {
        if (t0 != tid) {  // beyond the first two per thread (more than 64 tiles)
#pragma unroll
            for (int u = 0; u < 2; ++u)
                if (t0 + u * kConsumerThreads < np) v[u] = ld_tagged(&p.part_ms[base * kWarps + t0 + u * kConsumerThreads]);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int t = t0 + u * kConsumerThreads;
            if (t >= np) break;
            const ulonglong2 ms = has_epoch(v[u], ep) ? v[u] : part_ms_wait(p, base * kWarps + t, v[u], ep, deadline);
            ms_merge(m, s, __uint_as_float((uint32_t)ms.x), __uint_as_float((uint32_t)ms.y));
            if (score) above += __ldcg(&p.part_rank[base * kWarps + t]).x;
        }
    }
    {
        // the warp's maximum first, then one rescaled sum
        const uint32_t om = __reduce_max_sync(kFull, ord32(__fadd_rn(m, 0.0f)));
        const float Mw = unord32(om);
        float sc = (m > kNegInf) ? s * ex2((m - Mw) * kLog2e) : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sc += __shfl_xor_sync(kFull, sc, o);
        m = Mw;
        s = sc;
    }
    if (score) above = (int)__reduce_add_sync(kFull, (unsigned)above);
    // ---- natural: the warp column's 8 largest summary entries (lane r < 8
    // keeps entry r), and their threads' vectors, loaded now
    unsigned long long mine = 0ull;
    uint32_t cv[kCachedShares][4];  // the entries' values, kept for the completeness check
    uint4 pv[2];
    long long pv0[2];
    if (natural) {
        // a share's 4 entries are stored largest first; a lane with two tiles
        // (rows of more than 32 tiles) merges them into its 4 largest
        unsigned long long top[4] = {ca[0].x, ca[0].y, cb[0].x, cb[0].y};
#pragma unroll
        for (int i = 0; i < kCachedShares; ++i) {
            cv[i][0] = (uint32_t)(ca[i].x >> 32);
            cv[i][1] = (uint32_t)(ca[i].y >> 32);
            cv[i][2] = (uint32_t)(cb[i].x >> 32);
            cv[i][3] = (uint32_t)(cb[i].y >> 32);
        }
        if (lane + 32 < T) {
            const unsigned long long ent[4] = {ca[1].x, ca[1].y, cb[1].x, cb[1].y};
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                unsigned long long x = ent[r];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const unsigned long long hi = x > top[k] ? x : top[k], lo = x > top[k] ? top[k] : x;
                    top[k] = hi;
                    x = lo;
                }
            }
        }
        // knock out the largest head eight times; the winning lane writes its
        // entry (a lane holding more than 4 of the column's 8 largest gives
        // smaller ones instead: still 8 distinct entries, all the threshold needs)
        uint32_t hv = (uint32_t)(top[0] >> 32);
#pragma unroll
        for (int r = 0; r < kWarpTop; ++r) {
            const uint32_t vmax = __reduce_max_sync(kFull, hv);
            const unsigned b = __ballot_sync(kFull, hv == vmax);
            if (lane == __ffs(b) - 1) {
                sm.wsel[warp][r] = vmax != 0u ? top[0] : 0ull;
                sm.wtop[warp][r] = vmax;
                top[0] = top[1];
                top[1] = top[2];
                top[2] = top[3];
                top[3] = 0ull;
                hv = (uint32_t)(top[0] >> 32);
            }
        }
        __syncwarp();
        if (lane < kWarpTop) mine = sm.wsel[warp][lane];
        // lane l loads vectors 2*(l & 3) and 2*(l & 3) + 1 of entry l >> 2
        const unsigned long long pe = sm.wsel[warp][lane >> 2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int c = 2 * (lane & 3) + h;
            const uint32_t pos = (uint32_t)pe;
            pv0[h] = (long long)(pos >> 8) * TE + (long long)(c * kConsumerThreads + (int)(pos & 0xFFu)) * EPV;
            if (pe == 0ull || pv0[h] >= p.V) pv0[h] = p.V;
            pv[h] = make_uint4(0u, 0u, 0u, 0u);
            if (pv0[h] < p.V) pv[h] = __ldcs(reinterpret_cast<const uint4*>(rowp + pv0[h] * ELT));
        }
    }
    if (lane == 0) {
        sm.red_f[warp] = m;
        sm.red_f2[warp] = s;
        sm.red_i[warp] = above;
    }
    if (tid == 32) sm.xchosen = xc;
    cbar();
    rtrace(p, kTrRecA, row);
    // ---- every warp: lse from the 8 warps' partials (identical in every warp)
    float lse, xch;
    {
        const float mw = lane < kWarps ? sm.red_f[lane] : kNegInf;
        const float sw = lane < kWarps ? sm.red_f2[lane] : 0.0f;
        const float M = unord32(__reduce_max_sync(kFull, ord32(__fadd_rn(mw, 0.0f))));
        float t = (mw > kNegInf) ? sw * ex2((mw - M) * kLog2e) : 0.0f;
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) t += __shfl_xor_sync(kFull, t, o);
        const float S = __shfl_sync(kFull, t, 0);
        // lse = M + log(S); S >= 1 holds the maximum's own term, so logf(S) is
        // accurate to an ulp of a small number and the sum rounds once
        lse = M + logf(S);
        xch = chosen_is_max ? M : sm.xchosen;
        if (warp == 0 && lane == 0) {
            sm.lse = lse;
            sm.xchosen = xch;
            sm.rec[0] = chosen;
            sm.rec[1] = (chosen >= 0 && chosen < p.V) ? (int)__float_as_uint(logprob(xch, lse)) : (int)kUnusedBits;
            if (p.lse_out) p.lse_out[row] = lse;
        }
    }
    if (natural) {
        // theta: the 32nd largest of the 8 warps' 8 largest entry values (0:
        // fewer than 32 entries), by a bitonic sort of the 64 values, element
        // 2 * lane + h on lane `lane`, descending
        uint32_t a0 = sm.wtop[lane >> 2][2 * (lane & 3)], a1 = sm.wtop[lane >> 2][2 * (lane & 3) + 1];
#pragma unroll
        for (int k = 2; k <= 64; k <<= 1) {
#pragma unroll
            for (int j = k >> 1; j > 0; j >>= 1) {
                if (j == 1) {
                    // elements 2*lane and 2*lane + 1: the lower index keeps the larger in a descending block
                    const bool desc = ((2 * lane) & k) == 0;
                    const uint32_t hi = a0 > a1 ? a0 : a1, lo = a0 > a1 ? a1 : a0;
                    a0 = desc ? hi : lo;
                    a1 = desc ? lo : hi;
                } else {
                    const int pl = lane ^ (j >> 1);
                    const uint32_t b0 = __shfl_sync(kFull, a0, pl), b1 = __shfl_sync(kFull, a1, pl);
                    const bool lower = (lane & (j >> 1)) == 0;
                    const bool desc = ((2 * lane) & k) == 0;
                    const bool keep_hi = lower == desc;
                    a0 = keep_hi ? (a0 > b0 ? a0 : b0) : (a0 > b0 ? b0 : a0);
                    a1 = keep_hi ? (a1 > b1 ? a1 : b1) : (a1 > b1 ? b1 : a1);
                }
            }
        }
        const uint32_t th = __shfl_sync(kFull, a1, 15);  // element 31
        const float theta = th ? unord32(th) : kNegInf;
        if (warp == 0 && lane == 0) sm.theta_o = th;
        // this column's candidate threads must all be among the 8 loaded
        int cnt = 0;
        bool full = false;
#pragma unroll
        for (int i = 0; i < kCachedShares; ++i) {
#pragma unroll
            for (int r = 0; r < 4; ++r) cnt += (cv[i][r] != 0u && cv[i][r] >= th) ? 1 : 0;
            full |= cv[i][3] != 0u && cv[i][3] >= th;
        }
        const int loaded = (lane < kWarpTop && mine != 0ull && (uint32_t)(mine >> 32) >= th) ? 1 : 0;
        const bool slow = th == 0u || T > 32 * kCachedShares ||
                          __any_sync(kFull, full) ||
                          __reduce_add_sync(kFull, (unsigned)cnt) != __reduce_add_sync(kFull, (unsigned)loaded);
        if (slow) {
            if (lane == 0) sm.slow = 1;
        } else {
            // the prefetched lanes >= theta, as logprob keys (warp-aggregated append)
            int n = 0;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (pv0[h] < p.V) {
#pragma unroll
                    for (int e = 0; e < EPV; ++e) n += (pv0[h] + e < p.V && vec_elem<ELT>(pv[h], e) >= theta) ? 1 : 0;
                }
            }
            int incl = n;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int q = __shfl_up_sync(kFull, incl, o);
                if (lane >= o) incl += q;
            }
            int k0 = 0;
            if (lane == 31 && incl > 0) k0 = atomicAdd(&sm.n_keys, incl);
            int k = __shfl_sync(kFull, k0, 31) + incl - n;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (pv0[h] < p.V) {
#pragma unroll
                    for (int e = 0; e < EPV; ++e) {
                        const float y = vec_elem<ELT>(pv[h], e);
                        if (pv0[h] + e < p.V && y >= theta) {
                            if (k < kCandKeys) sm.ckeys[k] = lp_key(y, lse, (uint32_t)(pv0[h] + e));
                            ++k;
                        }
                    }
                }
            }
        }
    }
    if constexpr (SCORE) {
        if (warp == 0) {
            const float xt = xch;
            const float lp = logprob(xt, lse);
            const float xl = lp == lp ? score_limit(xt, lse, lp, lane) : xt;  // NaN: nothing is above
            if (lane == 0) sm.xlim = xl;
        }
    }
    cbar();
    rtrace(p, kTrRecB, row);
    if (natural) {
        const int keff = (long long)kc < p.V ? kc : (int)p.V;
        const Span whole = {0, T, 0, p.V};
        if (sm.slow) {
            if (tid == 0) sm.n_keys = 0;
            cbar();
            natural_record<ELT>(p, sm, row, base, whole, keff);
        } else {
            natural_rank<ELT>(p, sm, row, whole, keff, lse);
        }
    }
    rtrace(p, kTrRecC, row);
    if (ids && tid < kc) {
        int bits = (int)kUnusedBits;
        if (id >= 0 && id < p.V) {
            bits = (int)__float_as_uint(logprob(xi, lse));
        } else {
            atomicOr(p.status, kStatusBadId);
        }
        sm.rec[2 + 2 * tid] = id;
        sm.rec[3 + 2 * tid] = bits;
    }
    if constexpr (SCORE) {
        // logits in (xt, X]: above the target's but reported equal to it.  Only
        // a tile whose smallest logit above the target's is <= X holds any.
        const float xt = xch, X = sm.xlim;
        int corr = 0;
        for (int t = warp; t < T; t += kWarps) {
            const float mn = lane < kWarps ? __uint_as_float((uint32_t)__ldcg(&p.part_rank[(base + t) * kWarps + lane]).y)
                                           : kPosInf;
            if (!__any_sync(kFull, mn <= X)) continue;
            const long long t0e = (long long)t * tile_elems<ELT>();
            const long long remv = p.V - t0e;
            const int nvt = remv < tile_elems<ELT>() ? (int)remv : tile_elems<ELT>();
            for (int e = lane; e < nvt; e += 32) {
                const float x = load_logit<ELT>(p, row, t0e + e);
                corr += (x > xt && x <= X) ? 1 : 0;
            }
        }
        corr = (int)__reduce_add_sync(kFull, (unsigned)corr);
        if (lane == 0 && corr != 0) atomicAdd(&sm.corr, corr);
    }
    cbar();
    if constexpr (SCORE) {
        // record: target, its lp, rank, then the 20 alternatives
        int above_all = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) above_all += sm.red_i[w];
        int* out = p.score_records + (long long)row * kScoreWords;
        for (int w = tid; w < kScoreWords; w += kConsumerThreads)
            out[w] = w < 2 ? sm.rec[w] : w == 2 ? 1 + above_all - sm.corr : sm.rec[w - 1];
    } else {
        int* out = p.records + (long long)row * kRecordWords;
        for (int w = tid; w < kRecordWords; w += kConsumerThreads) out[w] = sm.rec[w];
    }
    cbar();
}

// Builds the records of the rows the stream kernel decides, while it runs.
// Launched after it with programmatic dependent launch, the grid is scheduled
// once every stream CTA has started: its CTAs take the multiprocessor room the
// stream grid leaves, then the room of each stream CTA that exits.  It does not
// wait for the stream grid to complete.  CTA b claims record tasks in order
// through a counter, waits until the claimed task's words carry the run's epoch
// (the decider wrote them after the row's last tile was counted), and builds
// the record; the tile partials it reads are run-tagged, or were performed
// before their tiles were counted.  A CTA stops once every group is decided
// and its claim is past the last task.
template <int ELT, bool SCORE>
__global__ void __launch_bounds__(kConsumerThreads, 3) lp_record_kernel(Params p) {
    __shared__ RecShared rs;
    __shared__ int4 s_task;  // the claimed task: (chosen, row, descriptor word | count << 16, group); row -1: none
    if (vload(&p.ctrl->abort) != 0u) {
        if (threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");  // completes after the stream grid
        return;
    }
    const uint32_t ep = vload(&p.ctrl->epoch);
    const unsigned long long deadline = globaltimer() + p.timeout_ns;
    unsigned long long* tr = p.trace != nullptr ? p.trace + ((size_t)p.trace_ctas * kTraceRoles) * p.trace_cap * 2 : nullptr;
    if (tr != nullptr && threadIdx.x == 0) {
        g_trace_n[3] = 0u;
        atomicMin(&tr[4], globaltimer());
    }
    rtrace(p, kTrKernel, 0);
    for (;;) {
        if (threadIdx.x == 0) {
            const unsigned i = atomicAdd(&p.ctrl->rec_claim, 1u);
            int4 t = make_int4(0, -1, 0, 0);
            for (;;) {
                if (i < (unsigned)p.rows) {
                    const ulonglong2 a = ld_tagged(&p.rec_tasks[2 * (size_t)i]);
                    const ulonglong2 b = ld_tagged(&p.rec_tasks[2 * (size_t)i + 1]);
                    if (has_epoch(a, ep) && has_epoch(b, ep)) {
                        t = make_int4((int)(uint32_t)a.x, (int)(uint32_t)a.y, (int)(uint32_t)b.x, (int)(uint32_t)b.y);
                        break;
                    }
                }
                // no task i once every group is decided and i is past the count:
                // the count is read after the outstanding groups are seen to be
                // none, and each decider appended its task before its group retired
                if (vload(&p.ctrl->outstanding) <= 0 && i >= vload(&p.ctrl->rec_count)) break;
                if (globaltimer() > deadline) {
                    atomicOr(p.status, kStatusTimeout);
                    break;
                }
                __nanosleep(128);
            }
            s_task = t;
        }
        __syncthreads();
        const int4 t = s_task;
        if (t.y < 0) break;
        rtrace(p, kTrRecStart, t.y);
        record_block<ELT, SCORE>(p, rs, t.y, t.w, t.x, t.z & 0x7FFF, t.z >> 16, ep, deadline);
        rtrace(p, kTrRecEnd, t.y);
    }
    if (tr != nullptr && threadIdx.x == 0) atomicMax(&tr[6], globaltimer());
    // this grid completes after the stream grid (it never waited for it):
    // whatever follows in the stream, the next run's prepare kernel included,
    // finds every kernel of the run done
    if (threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Test hook: each CTA holds `smem` bytes of shared memory (so no stream CTA
// fits beside it) and spins on the global timer for `ns`, then exits.
__global__ void lp_occupy_kernel(unsigned long long ns) {
    extern __shared__ unsigned char occ[];
    const unsigned long long t0 = globaltimer();
    if (threadIdx.x == 0) occ[0] = 0;
    while (globaltimer() - t0 < ns) __nanosleep(1000);
}

// ------------------------------------------------------------------ vocabulary-sharded records
//
// Source: "logprobs-design.md", the vocabulary-sharded speculative
// verification paragraph: each rank holds a vocabulary shard of the target
// logits; a first all-gather carries each shard's maximum and exponential mass
// (the global normalisation), a second the chosen token's raw logit from its
// owning rank and either the shard's best 32 sort keys or the selected ids' raw
// logits (256 words per position per rank); a final launch merges the gathered
// candidates into the same packed record.
//
// Here the shards are S column ranges of whole tiles of one block on one GPU:
// shard s of a row covers tiles [s*T/S, (s+1)*T/S).  Acceptance and the tile
// partials come from the stream kernel (on several GPUs that is the
// verification step, which decides the emitted prefix before the reduction).
// For record task i, shard s writes exchange 1 at x1[i*S + s] and exchange 2 at
// x2[(i*S + s)*256]; the kernels read another shard's payload only after the
// launch that wrote it has completed, as the all-gathers order them.

// Record task i, once the stream kernel has completed: (chosen, row, descriptor
// word | flags | count << 16, group).
__device__ __forceinline__ int4 load_task(const Params& p, unsigned i) {
    const ulonglong2 a = __ldcg(&p.rec_tasks[2 * (size_t)i]), b = __ldcg(&p.rec_tasks[2 * (size_t)i + 1]);
    return make_int4((int)(uint32_t)a.x, (int)(uint32_t)a.y, (int)(uint32_t)b.x, (int)(uint32_t)b.y);
}

__device__ __forceinline__ Span shard_span(const Params& p, int s, int S) {
    Span sp;
    sp.t0 = (int)((long long)s * p.T / S);
    sp.t1 = (int)((long long)(s + 1) * p.T / S);
    const long long te = p.elt == 2 ? tile_elems<2>() : tile_elems<4>();
    sp.v0 = (long long)sp.t0 * te;
    const long long e1 = (long long)sp.t1 * te;
    sp.v1 = e1 < p.V ? e1 : p.V;
    return sp;
}

// Exchange 1: warp s (< S) of the CTA of task i merges the (max, exp-sum)
// partials of shard s's tiles.
__global__ void __launch_bounds__(kConsumerThreads) lp_shard_stage1_kernel(Params p, int S, float2* x1) {
    const unsigned n = __ldcg(&p.ctrl->rec_count);
    const int lane = threadIdx.x & 31, s = threadIdx.x >> 5;
    if (s >= S || vload(&p.ctrl->abort) != 0u) return;
    for (unsigned i = blockIdx.x; i < n; i += gridDim.x) {
        const int row = load_task(p, i).y;
        const Span sp = shard_span(p, s, S);
        const long long base = (long long)row * p.T;
        float m = kNegInf, sum = 0.0f;
        for (int q = sp.t0 * kWarps + lane; q < sp.t1 * kWarps; q += 32) {
            const ulonglong2 ms = __ldcg(&p.part_ms[base * kWarps + q]);
            ms_merge(m, sum, __uint_as_float((uint32_t)ms.x), __uint_as_float((uint32_t)ms.y));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ms_merge(m, sum, __shfl_xor_sync(kFull, m, o), __shfl_xor_sync(kFull, sum, o));
        if (lane == 0) x1[(size_t)i * S + s] = make_float2(m, sum);
    }
}

// lse of task i from the gathered exchange 1 (every shard merges in the same
// order, so every shard gets the same bits).
__device__ __forceinline__ float shard_lse(const float2* x1, unsigned i, int S) {
    float M = kNegInf, T = 0.0f;
    for (int s = 0; s < S; ++s) {
        const float2 ms = __ldcg(&x1[(size_t)i * S + s]);
        ms_merge(M, T, ms.x, ms.y);
    }
    return M + logf(T);
}

// Exchange 2: CTA (i, s) writes shard s's 256-word payload of task i:
//   [0]           raw logit bits of the chosen token if the shard owns it, else NaN bits
//   natural rows: [1 + 2r], [2 + 2r] = (high, low) word of the shard's r-th best
//                 sort key (ord32(logprob) << 32 | ~id), r < 32, 0 = none
//   explicit ids: [1 + c] = raw logit bits of id c if the shard owns it, else NaN bits
template <int ELT>
__global__ void __launch_bounds__(kConsumerThreads, 3) lp_shard_stage2_kernel(Params p, int S, const float2* x1, int* x2) {
    __shared__ RecShared sm;
    const unsigned n = __ldcg(&p.ctrl->rec_count);
    if (vload(&p.ctrl->abort) != 0u) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (unsigned bi = blockIdx.x; bi < n * (unsigned)S; bi += gridDim.x) {
        const unsigned i = bi / S;
        const int s = (int)(bi % S);
        const int4 t = load_task(p, i);  // (chosen, row, descriptor word | flags | count << 16, group)
        const int row = t.y, chosen = t.x, g = t.w, dy = t.z & 0x7FFF, kc = t.z >> 16;
        const int mode = (dy >> 8) & 3, ids = (dy >> 12) & 1;
        const bool natural = !ids && mode == kModeNatural && kc > 0;
        const Span sp = shard_span(p, s, S);
        const long long base = (long long)row * p.T;
        int* out = x2 + ((size_t)i * S + s) * kShardWords;
        // each thread writes one word: the chosen logit, an id's logit, or the fill
        static_assert(kShardWords == kConsumerThreads, "one payload word per thread");
        {
            const int w = tid;
            int v = natural ? 0 : (int)kUnusedBits;
            if (w == 0) {
                v = (chosen >= sp.v0 && chosen < sp.v1) ? (int)__float_as_uint(load_logit<ELT>(p, row, chosen))
                                                         : (int)kUnusedBits;
            } else if (ids && w - 1 < kc) {
                const int id = __ldg(&p.token_ids[(long long)g * kMaxIds + (w - 1)]);
                v = (id >= sp.v0 && id < sp.v1) ? (int)__float_as_uint(load_logit<ELT>(p, row, id)) : (int)kUnusedBits;
            }
            out[w] = v;
        }
        if (tid == 0) {
            sm.n_thr = sm.n_sh = sm.n_keys = 0;
            sm.lse = shard_lse(x1, i, S);
        }
        if (natural) summary_top(p, sm, base, sp, warp, lane);
        cbar();
        if (natural) {
            if (warp == 0) {
                const uint32_t* wt = &sm.wtop[0][0];
                const uint32_t a = wt[lane], b = wt[lane + 32];
                int ra = 0, rb = 0;
#pragma unroll 8
                for (int j = 0; j < 64; ++j) {
                    const uint32_t v = wt[j];
                    ra += v > a || (v == a && j < lane);
                    rb += v > b || (v == b && j < lane + 32);
                }
                if (ra == 31) sm.theta_o = a;
                if (rb == 31) sm.theta_o = b;
            }
            for (int w = tid; w < 66; w += kConsumerThreads) sm.rec[w] = (w >= 2 && (w & 1) == 0) ? -1 : (int)kUnusedBits;
            cbar();
            const long long len = sp.v1 - sp.v0;
            natural_record<ELT>(p, sm, row, base, sp, len < 32 ? (int)len : 32);
            // the shard's best keys, from the pairs in rank order
            if (warp == 0) {
                const int id = sm.rec[2 + 2 * lane];
                const float lp = __uint_as_float((uint32_t)sm.rec[3 + 2 * lane]);
                const unsigned long long key =
                    id >= 0 ? ((unsigned long long)ord32(lp) << 32) | (unsigned long long)(~(uint32_t)id) : 0ull;
                out[1 + 2 * lane] = (int)(uint32_t)(key >> 32);
                out[2 + 2 * lane] = (int)(uint32_t)key;
            }
        }
        cbar();
    }
}

// Final merge: CTA of task i gathers the S payloads into the packed record.
__global__ void __launch_bounds__(kConsumerThreads) lp_shard_merge_kernel(Params p, int S, const float2* x1, const int* x2) {
    __shared__ unsigned long long lists[kMaxShards][32];
    __shared__ int rec[kRecordWords];
    __shared__ float lse_s;
    const unsigned n = __ldcg(&p.ctrl->rec_count);
    if (vload(&p.ctrl->abort) != 0u) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (unsigned i = blockIdx.x; i < n; i += gridDim.x) {
        const int4 t = load_task(p, i);
        const int row = t.y, chosen = t.x, dy = t.z & 0x7FFF, kc = t.z >> 16, g = t.w;
        const int mode = (dy >> 8) & 3, ids = (dy >> 12) & 1;
        const bool natural = !ids && mode == kModeNatural && kc > 0;
        const int* pay = x2 + (size_t)i * S * kShardWords;
        for (int w = tid; w < kRecordWords; w += kConsumerThreads) rec[w] = (w >= 2 && (w & 1) == 0) ? -1 : (int)kUnusedBits;
        if (tid == 0) lse_s = shard_lse(x1, i, S);
        if (natural && warp < S) {
            lists[warp][lane] = ((unsigned long long)(uint32_t)__ldcg(&pay[warp * kShardWords + 1 + 2 * lane]) << 32) |
                                (uint32_t)__ldcg(&pay[warp * kShardWords + 2 + 2 * lane]);
        }
        __syncthreads();
        const float lse = lse_s;
        if (tid == 0) {
            float xc = kNegInf;
            bool found = false;
            for (int s = 0; s < S; ++s) {
                const int w = __ldcg(&pay[s * kShardWords]);
                if ((uint32_t)w != kUnusedBits) {
                    xc = __uint_as_float((uint32_t)w);
                    found = true;
                }
            }
            rec[0] = chosen;
            rec[1] = found ? (int)__float_as_uint(logprob(xc, lse)) : (int)kUnusedBits;
            if (p.lse_out) p.lse_out[row] = lse;
        }
        if (natural && warp == 0) {
            unsigned long long r = lists[0][lane];
            for (int s = 1; s < S; ++s) r = merge_lists(r, lists[s][lane], lane);
            const int keff = (long long)kc < p.V ? kc : (int)p.V;
            if (lane < keff && r != 0ull) {
                rec[2 + 2 * lane] = (int)key_id(r);
                rec[3 + 2 * lane] = (int)__float_as_uint(key_value(r));
            }
        }
        if (ids && tid < kc) {
            const int id = __ldg(&p.token_ids[(long long)g * kMaxIds + tid]);
            int bits = (int)kUnusedBits;
            for (int s = 0; s < S; ++s) {
                const int w = __ldcg(&pay[s * kShardWords + 1 + tid]);
                if ((uint32_t)w != kUnusedBits) bits = (int)__float_as_uint(logprob(__uint_as_float((uint32_t)w), lse));
            }
            if (id < 0 || id >= p.V) atomicOr(p.status, kStatusBadId);
            rec[2 + 2 * tid] = id;
            rec[3 + 2 * tid] = bits;
        }
        __syncthreads();
        int* o = p.records + (long long)row * kRecordWords;
        for (int w = tid; w < kRecordWords; w += kConsumerThreads) o[w] = rec[w];
        __syncthreads();
    }
}

template <int ELT>
constexpr int stream_smem_bytes() {
    return StageCfg<ELT>::kStages * kTileBytes + (int)sizeof(Shared) + (int)kStageAlign;
}

}  // namespace

cudaError_t query_launch_cfg(int dtype, LaunchCfg* cfg) {
    int dev = 0, sms = 0, occ = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    // both instances (generation, prompt scoring) have the same launch shape
    if (dtype == 1) {
        const int smem = stream_smem_bytes<2>();
        e = cudaFuncSetAttribute(lp_stream_kernel<2, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(lp_stream_kernel<2, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, lp_stream_kernel<2, false>, kThreads, smem);
        cfg->smem_bytes = smem;
    } else {
        const int smem = stream_smem_bytes<4>();
        e = cudaFuncSetAttribute(lp_stream_kernel<4, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(lp_stream_kernel<4, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, lp_stream_kernel<4, false>, kThreads, smem);
        cfg->smem_bytes = smem;
    }
    if (e != cudaSuccess) return e;
    cfg->grid = sms * (occ > 0 ? occ : 1);
    cfg->sms = sms;
    return cudaSuccess;
}

cudaError_t launch_occupy(int ctas, unsigned long long ns, cudaStream_t stream) {
    int dev = 0, smem = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(lp_occupy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    lp_occupy_kernel<<<ctas, 32, smem, stream>>>(ns);
    return cudaGetLastError();
}

cudaError_t launch_shard_records(const Params& p, int dtype, const LaunchCfg& cfg, int S, float2* x1, int* x2,
                                 cudaStream_t stream) {
    int grid = cfg.sms * 3;
    if (grid > p.rows) grid = p.rows > 0 ? p.rows : 1;
    lp_shard_stage1_kernel<<<grid, kConsumerThreads, 0, stream>>>(p, S, x1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    int grid2 = cfg.sms * 3;
    if ((long long)grid2 > (long long)p.rows * S) grid2 = p.rows * S > 0 ? p.rows * S : 1;
    if (dtype == 1) lp_shard_stage2_kernel<2><<<grid2, kConsumerThreads, 0, stream>>>(p, S, x1, x2);
    else lp_shard_stage2_kernel<4><<<grid2, kConsumerThreads, 0, stream>>>(p, S, x1, x2);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    lp_shard_merge_kernel<<<grid, kConsumerThreads, 0, stream>>>(p, S, x1, x2);
    return cudaGetLastError();
}

cudaError_t launch_epilogue(const Params& p_in, int dtype, const LaunchCfg& cfg, cudaStream_t stream, bool records) {
    long long work = (long long)p_in.rows * p_in.T;
    // stream-CTA slots left to the record kernel from the start
    int grid = cfg.grid - (records ? (LP_RECORD_SLOTS < cfg.grid / 2 ? LP_RECORD_SLOTS : cfg.grid / 2) : 0);
    if (work < grid) grid = work > 0 ? (int)work : 1;
    Params p = p_in;
    p.stream_grid = grid;
    p.build_records = records ? 1 : 0;
    lp_prepare_kernel<<<1, LP_PREP_THREADS, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(grid);
    lc.blockDim = dim3(kThreads);
    lc.dynamicSmemBytes = cfg.smem_bytes;
    lc.stream = stream;
    lc.attrs = attr;
    lc.numAttrs = 1;
    const bool score = p.targets != nullptr;
    if (dtype == 1) {
        e = score ? cudaLaunchKernelEx(&lc, lp_stream_kernel<2, true>, p) : cudaLaunchKernelEx(&lc, lp_stream_kernel<2, false>, p);
    } else {
        e = score ? cudaLaunchKernelEx(&lc, lp_stream_kernel<4, true>, p) : cudaLaunchKernelEx(&lc, lp_stream_kernel<4, false>, p);
    }
    if (e != cudaSuccess || !records) return e;
    // records: a persistent grid, one CTA per stream-CTA slot of the device
    // (the ones the stream grid leaves start at once, the others as stream CTAs
    // exit), at most one per row
    int rgrid = cfg.grid;
    if (rgrid > p.rows) rgrid = p.rows;
    if (rgrid < 1) rgrid = 1;
    cudaLaunchConfig_t rc = {};
    rc.gridDim = dim3(rgrid);
    rc.blockDim = dim3(kConsumerThreads);
    rc.dynamicSmemBytes = 0;
    rc.stream = stream;
    rc.attrs = attr;
    rc.numAttrs = 1;
    if (dtype == 1) {
        return score ? cudaLaunchKernelEx(&rc, lp_record_kernel<2, true>, p) : cudaLaunchKernelEx(&rc, lp_record_kernel<2, false>, p);
    }
    return score ? cudaLaunchKernelEx(&rc, lp_record_kernel<4, true>, p) : cudaLaunchKernelEx(&rc, lp_record_kernel<4, false>, p);
}

}  // namespace lp
