// lp_kernels.cu -- sm_103a kernels of the logprob / greedy-acceptance epilogue.
//
// Two launches per run, both on the caller's stream:
//
//  lp_prepare_kernel (1 CTA)
//    validates group_indptr, resolves each group's request (natural
//    alternatives, explicit ids or argmax only), finishes groups that need no
//    logits, resets the per-row work counters and writes the depth-0 work
//    queue: row 0 of every group that must be read.
//
//  lp_stream_kernel (persistent, PDL-overlapped with the prepare kernel)
//    one producer warp per CTA takes (row, tile) work items from a device FIFO
//    and streams each 8192-element vocabulary tile into a shared-memory stage
//    with a TMA bulk copy (cp.async.bulk, mbarrier completion, L2 evict-first);
//    eight compute warps reduce the tile: FP32 max, exp-sum (ex2) relative to
//    the tile max, the argmax key and, for rows that report natural
//    alternatives, the tile's best 32 packed sort keys
//        key = ord32(x) << 32 | (0xFFFFFFFF - id),
//    ord32 being the monotone float -> uint map with -0 folded into +0.
//    The CTA that finishes a row's last tile merges the row: argmax -> greedy
//    acceptance (on acceptance the next row of the group is appended to the
//    FIFO, so rows past the accepted prefix are never read), then
//    lse = M + log(sum s_t exp(m_t - M)), the chosen token's logprob, the
//    top-K natural alternatives or the explicit-id gather, and the 258-word
//    record.
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

struct Shared {
    uint64_t full[4];
    uint64_t empty[4];
    int4 info[4];
    unsigned long long cand[kCandCap];
    unsigned long long top[32];
    unsigned long long lists[8][32];
    unsigned long long red_u64[8];
    double red_d[8];
    float red_f[8];
    float red_f2[8];
    float theta_w[8];
    int red_i[8];
    int ncand;
    int last;
    int chosen;
    int pad0;
    int rec[kRecordWords + 2];
};

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

__device__ __forceinline__ float block_sum_f(float v, Shared& sm, int lane, int warp) {
    v = warp_sum_f(v);
    if (lane == 0) sm.red_f[warp] = v;
    cbar();
    float r = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) r += sm.red_f[i];
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

__device__ __forceinline__ unsigned long long block_max_u64(unsigned long long v, Shared& sm, int lane, int warp) {
    v = warp_max_u64(v);
    if (lane == 0) sm.red_u64[warp] = v;
    cbar();
    unsigned long long r = sm.red_u64[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) r = sm.red_u64[i] > r ? sm.red_u64[i] : r;
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

// ---- tile element access
//
// Full tiles: thread i owns the 16-byte vectors c*256 + i (c = 0..NCH-1), so
// element k = c*EPV + s of the thread is tile element (c*256 + i)*EPV + s.
// Partial tiles (the last tile of a row): element k of thread i is tile element
// k*256 + i, masked beyond the valid count.  Both orders are ascending in k.

template <int ELT>
struct TileLayout {
    static constexpr int EPV = 16 / ELT;          // elements per 16-byte vector
    static constexpr int NCH = 32 / EPV;          // vectors per thread
};

template <int ELT>
__device__ __forceinline__ int tile_elem_id(bool full, int k, int tid) {
    using L = TileLayout<ELT>;
    return full ? ((k / L::EPV) * kConsumerThreads + tid) * L::EPV + (k % L::EPV) : k * kConsumerThreads + tid;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <int ELT>
__device__ __forceinline__ void load_tile(const unsigned char* stage, bool full, int nv, int tid, float (&x)[32]) {
    using L = TileLayout<ELT>;
    if (full) {
#pragma unroll
        for (int c = 0; c < L::NCH; ++c) {
            const uint4 v = *reinterpret_cast<const uint4*>(stage + (size_t)(c * kConsumerThreads + tid) * 16);
            if constexpr (ELT == 4) {
                x[c * 4 + 0] = __uint_as_float(v.x);
                x[c * 4 + 1] = __uint_as_float(v.y);
                x[c * 4 + 2] = __uint_as_float(v.z);
                x[c * 4 + 3] = __uint_as_float(v.w);
            } else {
                x[c * 8 + 0] = bf16_lo(v.x);
                x[c * 8 + 1] = bf16_hi(v.x);
                x[c * 8 + 2] = bf16_lo(v.y);
                x[c * 8 + 3] = bf16_hi(v.y);
                x[c * 8 + 4] = bf16_lo(v.z);
                x[c * 8 + 5] = bf16_hi(v.z);
                x[c * 8 + 6] = bf16_lo(v.w);
                x[c * 8 + 7] = bf16_hi(v.w);
            }
        }
    } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            const int e = k * kConsumerThreads + tid;
            float v = kNegInf;
            if (e < nv) {
                if constexpr (ELT == 4) {
                    v = reinterpret_cast<const float*>(stage)[e];
                } else {
                    v = __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const unsigned short*>(stage)[e]) << 16);
                }
            }
            x[k] = v;
        }
    }
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

// ------------------------------------------------------------------ prepare

__global__ void __launch_bounds__(1024) lp_prepare_kernel(Params p) {
    asm volatile("griddepcontrol.launch_dependents;");
    __shared__ int s_warp[32];
    __shared__ int s_total;
    __shared__ int s_base;
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    for (int r = tid; r < p.rows; r += blockDim.x) {
        p.ticket[r] = 0;
        p.done[r] = 0;
        p.queue[r] = -1;
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
            p.ctrl->q_head = 0u;
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
        int need = 0;
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
        if (need) p.queue[s_base + s_warp[warp] + pos_in_warp] = g << 4;
        __syncthreads();
        if (tid == 0) s_base += s_total;
        __syncthreads();
    }
    if (st) atomicOr(p.status, st);
    if (tid == 0) {
        p.ctrl->q_head = 0u;
        p.ctrl->q_tail = static_cast<unsigned>(s_base);
        p.ctrl->outstanding = s_base;
        p.ctrl->abort = 0u;
    }
}

// ------------------------------------------------------------------ producer

template <int ELT>
__device__ void producer_loop(const Params& p, Shared& sm, unsigned char* stages, unsigned long long t0) {
    constexpr int S = StageCfg<ELT>::kStages;
    constexpr int TILE_BYTES = kTileElems * ELT;
    const unsigned long long deadline = t0 + p.timeout_ns;
    const uint64_t policy = evict_first_policy();
    Ctrl* ctrl = p.ctrl;
    const int T = p.T;
    int stage = 0;
    uint32_t phase = 0;
    int cur_entry = -1, cur_row = 0, cur_mode = 0;
    unsigned cur_pos = 0;
    bool stop = false;
    while (!stop) {
        int4 item = make_int4(0, 0, -1, 0);
        if (p.debug_flags & kDebugForceTimeout) {
            // Test hook: wait on a flag that nothing sets, until the limit.
            while (vload(&ctrl->never) == 0u) {
                if (globaltimer() > deadline) break;
                __nanosleep(1000);
            }
            atomicOr(p.status, kStatusTimeout);
            stop = true;
        } else {
            for (;;) {
                if (cur_entry >= 0) {
                    const int t = atomicAdd(&p.ticket[cur_row], 1);
                    if (t < T) {
                        item = make_int4(cur_row, t, cur_entry, cur_mode);
                        break;
                    }
                    atomicCAS(&ctrl->q_head, cur_pos, cur_pos + 1u);
                    cur_entry = -1;
                }
                const unsigned h = vload(&ctrl->q_head);
                const unsigned tl = vload(&ctrl->q_tail);
                if (h < tl) {
                    int e = vload(&p.queue[h]);
                    for (uint32_t i = 0; e < 0; ++i) {  // reserved, not yet published
                        if ((i & 63u) == 63u && globaltimer() > deadline) break;
                        e = vload(&p.queue[h]);
                    }
                    if (e < 0) {
                        atomicOr(p.status, kStatusTimeout);
                        stop = true;
                        break;
                    }
                    const int4 d = __ldcg(&p.gdesc[e >> 4]);
                    cur_entry = e;
                    cur_pos = h;
                    cur_row = d.x + (e & 15);
                    cur_mode = (d.y >> 8) & 3;
                    continue;
                }
                if (vload(&ctrl->outstanding) <= 0) {
                    stop = true;
                    break;
                }
                if (globaltimer() > deadline) {
                    atomicOr(p.status, kStatusTimeout);
                    stop = true;
                    break;
                }
                __nanosleep(32);
            }
        }
        if (!mbar_wait(&sm.empty[stage], phase ^ 1u, deadline)) {
            atomicOr(p.status, kStatusTimeout);
            return;
        }
        sm.info[stage] = item;
        if (item.z < 0) {
            mbar_arrive(&sm.full[stage]);
            return;
        }
        const long long tbase = (long long)item.y * kTileElems;
        const long long rem = p.V - tbase;
        const int nv = rem < kTileElems ? (int)rem : kTileElems;
        const uint32_t bytes = (static_cast<uint32_t>(nv * ELT) + 15u) & ~15u;
        const unsigned char* src =
            reinterpret_cast<const unsigned char*>(p.logits) + ((long long)item.x * p.Vp + tbase) * ELT;
        mbar_arrive_expect_tx(&sm.full[stage], bytes);
        bulk_load(stages + (size_t)stage * TILE_BYTES, src, bytes, &sm.full[stage], policy);
        if (++stage == S) {
            stage = 0;
            phase ^= 1u;
        }
    }
}

// ------------------------------------------------------------------ tile: exact slow top-32

// Exact top-32 keys of a tile when the candidate buffer overflowed (massive
// ties): the 32nd largest value v is found by walking distinct values down from
// the maximum; the result is every lane above v plus the smallest ids equal to v.
template <int ELT>
__device__ __noinline__ void tile_top32_slow(const unsigned char* stage, bool full, int nv, long long tbase,
                                             Shared& sm) {
    using L = TileLayout<ELT>;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float x[32];
    load_tile<ELT>(stage, full, nv, tid, x);
    float v = __builtin_huge_valf();
    int cnt_ge = 0;
    for (int it = 0; it < 33; ++it) {
        float loc = kNegInf;
#pragma unroll
        for (int k = 0; k < 32; ++k) loc = (x[k] < v && x[k] > loc) ? x[k] : loc;
        const float vn = block_max_f(loc, sm, lane, warp);
        if (!(vn > kNegInf)) break;  // no value left below v
        v = vn;
        int c = 0;
#pragma unroll
        for (int k = 0; k < 32; ++k) c += (x[k] >= v && x[k] > kNegInf) ? 1 : 0;
        cnt_ge = block_sum_i(c, sm, lane, warp);
        if (cnt_ge >= 32) break;
    }
    int c = 0;
#pragma unroll
    for (int k = 0; k < 32; ++k) c += (x[k] > v && x[k] > kNegInf) ? 1 : 0;
    const int cnt_gt = block_sum_i(c, sm, lane, warp);
    const int take = (cnt_ge < 32 ? cnt_ge : 32);
    const int need_eq = take - cnt_gt;
    if (tid == 0) sm.ncand = 0;
    cbar();
#pragma unroll
    for (int k = 0; k < 32; ++k) {
        if (x[k] > v && x[k] > kNegInf) {
            const int pos = atomicAdd(&sm.ncand, 1);
            if (pos < 32) sm.cand[pos] = make_key(x[k], (uint32_t)(tbase + tile_elem_id<ELT>(full, k, tid)));
        }
    }
    // lanes equal to v, in ascending id order, until need_eq are taken
    const int NQ = full ? L::NCH : 32;
    const int SPQ = full ? L::EPV : 1;
    int got = 0;
    for (int q = 0; q < NQ && got < need_eq; ++q) {
        int mine = 0;
        for (int s = 0; s < SPQ; ++s) {
            const int k = q * SPQ + s;
            float xv = kNegInf;
#pragma unroll
            for (int kk = 0; kk < 32; ++kk) xv = (kk == k) ? x[kk] : xv;
            mine += (xv == v && xv > kNegInf) ? 1 : 0;
        }
        int total = 0;
        int before = block_excl_scan_i(mine, &total, sm, lane, warp);
        for (int s = 0; s < SPQ; ++s) {
            const int k = q * SPQ + s;
            float xv = kNegInf;
#pragma unroll
            for (int kk = 0; kk < 32; ++kk) xv = (kk == k) ? x[kk] : xv;
            if (xv == v && xv > kNegInf) {
                const int pos = got + before;
                if (pos < need_eq) sm.cand[cnt_gt + pos] = make_key(xv, (uint32_t)(tbase + tile_elem_id<ELT>(full, k, tid)));
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
        sm.top[rank] = key;
    }
    if (tid >= n && tid < 32) sm.top[tid] = 0ull;
    cbar();
}

// ------------------------------------------------------------------ merge

template <int ELT>
__device__ __noinline__ void merge_row(const Params& p, Shared& sm, int row, int entry) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = entry >> 4, j = entry & 15;
    const int4 d = __ldcg(&p.gdesc[g]);
    const int r0 = d.x, k = d.y & 0xFF, mode = (d.y >> 8) & 3, ids = (d.y >> 12) & 1, req = (d.y >> 13) & 1;
    const int kc = d.z, samp = d.w;
    const int T = p.T;
    const long long base = (long long)row * T;

    unsigned long long bk = 0;
    float tm = kNegInf;
    for (int t = tid; t < T; t += kConsumerThreads) {
        const unsigned long long key = __ldcg(&p.part_keys[(base + t) * kKeysPerTile]);
        bk = key > bk ? key : bk;
        if (req) tm = fmaxf(tm, __ldcg(&p.part_ms[base + t]).x);
    }
    bk = block_max_u64(bk, sm, lane, warp);
    const uint32_t amax = key_id(bk);

    if (tid == 0) {
        const int chosen = (k == 0 && samp >= 0) ? samp : (int)amax;
        p.emitted[row] = chosen;
        const bool accept = (j < k) && (p.drafts[row] == (int)amax);
        if (accept) {
            const unsigned pos = atomicAdd(&p.ctrl->q_tail, 1u);
            vstore(&p.queue[pos], (g << 4) | (j + 1));
        } else {
            p.accepted[g] = j;
            for (int jj = j + 1; jj <= k; ++jj) p.emitted[r0 + jj] = -1;
            __threadfence();
            atomicSub(&p.ctrl->outstanding, 1);
        }
        if (req && chosen >= p.V) atomicOr(p.status, kStatusBadToken);
        sm.chosen = chosen;
    }
    if (!req) {
        cbar();
        return;
    }
    for (int w = tid; w < kRecordWords; w += kConsumerThreads)
        sm.rec[w] = (w >= 2 && (w & 1) == 0) ? -1 : (int)kUnusedBits;

    // lse = M + log(sum_t s_t exp(m_t - M)); the few per-tile terms are combined
    // in FP64 and the result is rounded once to FP32
    const float M = block_max_f(tm, sm, lane, warp);
    double ps = 0.0;
    for (int t = tid; t < T; t += kConsumerThreads) {
        const float2 ms = __ldcg(&p.part_ms[base + t]);
        ps += (double)ms.y * exp((double)ms.x - (double)M);
    }
    const double S = block_sum_d(ps, sm, lane, warp);  // has barriers: rec defaults and sm.chosen visible
    const float lse = __double2float_rn((double)M + log(S));
    const int chosen = sm.chosen;
    if (tid == 0) {
        sm.rec[0] = chosen;
        sm.rec[1] = (chosen >= 0 && chosen < p.V) ? (int)__float_as_uint(logprob(load_logit<ELT>(p, row, chosen), lse))
                                                  : (int)kUnusedBits;
        if (p.lse_out) p.lse_out[row] = lse;
    }
    if (ids) {
        for (int i = tid; i < kc; i += kConsumerThreads) {
            const int id = p.token_ids[(long long)g * kMaxIds + i];
            int bits = (int)kUnusedBits;
            if (id >= 0 && id < p.V) {
                bits = (int)__float_as_uint(logprob(load_logit<ELT>(p, row, id), lse));
            } else {
                atomicOr(p.status, kStatusBadId);
            }
            sm.rec[2 + 2 * i] = id;
            sm.rec[3 + 2 * i] = bits;
        }
    } else if (mode == kModeNatural && kc > 0) {
        // global raw top-32: each warp merges its tiles, warp 0 merges the warps
        unsigned long long r = 0;
        for (int t = warp; t < T; t += 8) {
            const unsigned long long nk = __ldcg(&p.part_keys[(base + t) * kKeysPerTile + lane]);
            const unsigned long long rev = __shfl_sync(kFull, nk, 31 - lane);
            r = warp_bitonic_clean_desc(rev > r ? rev : r, lane);
        }
        sm.lists[warp][lane] = r;
        cbar();
        if (warp == 0) {
            r = sm.lists[0][lane];
#pragma unroll 1
            for (int w = 1; w < 8; ++w) {
                const unsigned long long o = sm.lists[w][31 - lane];
                r = warp_bitonic_clean_desc(o > r ? o : r, lane);
            }
            const bool real = r != 0ull;
            const float lp = real ? logprob(key_value(r), lse) : kNegInf;
            const int keff = (long long)kc < p.V ? kc : (int)p.V;
            const float Lk = __shfl_sync(kFull, lp, keff - 1);
            const float lp31 = __shfl_sync(kFull, lp, 31);
            const bool fallback = (p.V > 32) && (lp31 == Lk);
            const unsigned long long key2 =
                real ? ((static_cast<unsigned long long>(ord32(lp)) << 32) | (r & 0xFFFFFFFFull)) : 0ull;
            const unsigned long long sorted = warp_sort_desc(key2, lane);
            const int c_gt = fallback ? __popc(__ballot_sync(kFull, real && lp > Lk)) : keff;
            if (lane < c_gt) {
                sm.rec[2 + 2 * lane] = (int)key_id(sorted);
                sm.rec[3 + 2 * lane] = (int)__float_as_uint(key_value(sorted));
            }
            if (fallback) {
                // lanes with logprob == Lk, smallest ids first, tile by tile
                const int need = keff - c_gt;
                const unsigned lbits = __float_as_uint(Lk);
                int got = 0;
                for (int t = 0; t < T && got < need; ++t) {
                    const long long t0e = (long long)t * kTileElems;
                    const long long remv = p.V - t0e;
                    const int nvt = remv < kTileElems ? (int)remv : kTileElems;
                    const unsigned long long kmin = __ldcg(&p.part_keys[(base + t) * kKeysPerTile + 31]);
                    const bool hid = nvt > 32 && kmin != 0ull && logprob(key_value(kmin), lse) == Lk;
                    if (hid) {
                        for (int e0 = 0; e0 < nvt && got < need; e0 += 32) {
                            const int e = e0 + lane;
                            const bool m = e < nvt && logprob(load_logit<ELT>(p, row, t0e + e), lse) == Lk;
                            const unsigned b = __ballot_sync(kFull, m);
                            const int before = __popc(b & ((1u << lane) - 1u));
                            if (m && got + before < need) {
                                sm.rec[2 + 2 * (c_gt + got + before)] = (int)(t0e + e);
                                sm.rec[3 + 2 * (c_gt + got + before)] = (int)lbits;
                            }
                            got += __popc(b);
                        }
                    } else {
                        const unsigned long long key = __ldcg(&p.part_keys[(base + t) * kKeysPerTile + lane]);
                        const bool m = key != 0ull && logprob(key_value(key), lse) == Lk;
                        // ascending ids: sort the complement descending
                        const uint32_t inv = m ? ~key_id(key) : 0u;
                        const uint32_t sorted_inv = warp_sort_desc(inv, lane);
                        const int cnt = __popc(__ballot_sync(kFull, m));
                        if (lane < cnt && got + lane < need) {
                            sm.rec[2 + 2 * (c_gt + got + lane)] = (int)(~sorted_inv);
                            sm.rec[3 + 2 * (c_gt + got + lane)] = (int)lbits;
                        }
                        got += cnt;
                    }
                }
            }
        }
    }
    cbar();
    int* out = p.records + (long long)row * kRecordWords;
    for (int w = tid; w < kRecordWords; w += kConsumerThreads) out[w] = sm.rec[w];
    cbar();
}

// ------------------------------------------------------------------ consumer

template <int ELT>
__device__ void consumer_loop(const Params& p, Shared& sm, unsigned char* stages, unsigned long long t0) {
    constexpr int S = StageCfg<ELT>::kStages;
    constexpr int TILE_BYTES = kTileElems * ELT;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned long long deadline = t0 + p.timeout_ns;
    const int T = p.T;
    int stage = 0;
    uint32_t phase = 0;
    for (;;) {
        // every compute thread leaves together if any of them ran out of time
        const bool late = !mbar_wait(&sm.full[stage], phase, deadline);
        if (cbar_or(late)) {
            if (tid == 0) atomicOr(p.status, kStatusTimeout);
            return;
        }
        const int4 info = sm.info[stage];
        if (info.z < 0) return;
        const unsigned char* sp = stages + (size_t)stage * TILE_BYTES;
        const int row = info.x, tile = info.y, entry = info.z, mode = info.w;
        const long long tbase = (long long)tile * kTileElems;
        const long long rem = p.V - tbase;
        const int nv = rem < kTileElems ? (int)rem : kTileElems;
        const bool full = nv == kTileElems;

        float x[32];
        load_tile<ELT>(sp, full, nv, tid, x);
        float m = x[0];
#pragma unroll
        for (int k = 1; k < 32; ++k) m = fmaxf(m, x[k]);

        const long long slot = (long long)row * T + tile;
        unsigned long long tile_key = 0;
        float M = 0.0f, ssum = 0.0f;

        if (mode == kModeNatural) {
            // threshold: min over warps of the warp's 4th largest thread maximum;
            // at least 32 lanes of the tile are >= theta
            const float sorted = warp_sort_desc(m, lane);
            if (lane == 0) sm.red_f[warp] = sorted;
            if (lane == 3) sm.theta_w[warp] = sorted;
            if (tid == 0) sm.ncand = 0;
            cbar();
            M = sm.red_f[0];
            float theta = sm.theta_w[0];
#pragma unroll
            for (int w = 1; w < 8; ++w) {
                M = fmaxf(M, sm.red_f[w]);
                theta = fminf(theta, sm.theta_w[w]);
            }
            // exp(x - M) = 2^(x*log2e - mb_hi - mb_lo); mb_lo (the rounding residual of
            // M*log2e) is folded in once per tile, so large |M| costs no accuracy
            const float mb = M * kLog2e;
            const float mb_lo = fmaf(M, kLog2e, -mb);
            float s = 0.0f;
#pragma unroll
            for (int k = 0; k < 32; ++k) s += ex2(fmaf(x[k], kLog2e, -mb));
            if (m >= theta && m > kNegInf) {
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    if (x[k] >= theta && x[k] > kNegInf) {
                        const int pos = atomicAdd(&sm.ncand, 1);
                        if (pos < kCandCap) sm.cand[pos] = make_key(x[k], (uint32_t)(tbase + tile_elem_id<ELT>(full, k, tid)));
                    }
                }
            }
            s = warp_sum_f(s);
            if (lane == 0) sm.red_f2[warp] = s;
            cbar();
            const int n = sm.ncand;
            ssum = 0.0f;
#pragma unroll
            for (int w = 0; w < 8; ++w) ssum += sm.red_f2[w];
            ssum *= ex2(-mb_lo);
            if (n <= kCandCap) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.empty[stage]);
                if (tid < n) {
                    const unsigned long long key = sm.cand[tid];
                    int rank = 0;
                    for (int u = 0; u < n; ++u) rank += sm.cand[u] > key ? 1 : 0;
                    if (rank < 32) sm.top[rank] = key;
                }
                if (tid >= n && tid < 32) sm.top[tid] = 0ull;
                cbar();
            } else {
                tile_top32_slow<ELT>(sp, full, nv, tbase, sm);
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.empty[stage]);
            }
            if (warp == 0) {
                p.part_keys[slot * kKeysPerTile + lane] = sm.top[lane];
                if (lane == 0) p.part_ms[slot] = make_float2(M, ssum);
            }
        } else {
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[stage]);
            // argmax key: first lane of the thread's maximum, then the block max
            unsigned long long tkey = 0;
            if (m > kNegInf) {
                int kf = 31;
#pragma unroll
                for (int k = 31; k >= 0; --k) kf = (x[k] == m) ? k : kf;
                tkey = make_key(m, (uint32_t)(tbase + tile_elem_id<ELT>(full, kf, tid)));
            }
            tkey = warp_max_u64(tkey);
            if (lane == 0) sm.red_u64[warp] = tkey;
            if (mode == kModeLse) {
                M = block_max_f(m, sm, lane, warp);  // barriers also publish red_u64
                const float mb = M * kLog2e;
                const float mb_lo = fmaf(M, kLog2e, -mb);
                float s = 0.0f;
#pragma unroll
                for (int k = 0; k < 32; ++k) s += ex2(fmaf(x[k], kLog2e, -mb));
                s = warp_sum_f(s) * ex2(-mb_lo);
                if (lane == 0) sm.red_f2[warp] = s;
            }
            cbar();
            if (warp == 0) {
                tile_key = sm.red_u64[0];
#pragma unroll
                for (int w = 1; w < 8; ++w) tile_key = sm.red_u64[w] > tile_key ? sm.red_u64[w] : tile_key;
                ssum = 0.0f;
                if (mode == kModeLse) {
#pragma unroll
                    for (int w = 0; w < 8; ++w) ssum += sm.red_f2[w];
                }
                if (lane == 0) {
                    p.part_keys[slot * kKeysPerTile] = tile_key;
                    p.part_ms[slot] = make_float2(M, ssum);
                }
            }
        }
        // publish the tile; the CTA finishing a row's last tile merges it
        if (warp == 0) {
            __threadfence();
            __syncwarp();
            if (lane == 0) {
                const int old = atomicAdd(&p.done[row], 1);
                __threadfence();
                sm.last = (old == T - 1) ? 1 : 0;
            }
        }
        cbar();
        if (sm.last) merge_row<ELT>(p, sm, row, entry);
        cbar();
        if (++stage == S) {
            stage = 0;
            phase ^= 1u;
        }
    }
}

template <int ELT>
__global__ void __launch_bounds__(kThreads, StageCfg<ELT>::kMinBlocks) lp_stream_kernel(Params p) {
    constexpr int S = StageCfg<ELT>::kStages;
    constexpr int TILE_BYTES = kTileElems * ELT;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* stages = smem_raw;
    Shared& sm = *reinterpret_cast<Shared*>(smem_raw + (size_t)S * TILE_BYTES);
    const int tid = threadIdx.x;
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kConsumerThreads / 32);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (vload(&p.ctrl->abort) != 0u) return;
    const unsigned long long t0 = globaltimer();
    if (tid >= kConsumerThreads) {
        if (tid == kConsumerThreads) producer_loop<ELT>(p, sm, stages, t0);
        return;
    }
    consumer_loop<ELT>(p, sm, stages, t0);
}

template <int ELT>
constexpr int stream_smem_bytes() {
    return StageCfg<ELT>::kStages * kTileElems * ELT + (int)sizeof(Shared);
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
