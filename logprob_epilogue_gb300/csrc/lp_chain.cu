// lp_chain.cu -- sm_103a kernel of stochastic chain verification.
//
// Source: "mtp-design.md", section "Sampling correctness": a draft drawn from
// the draft law q is accepted with probability min(1, p/q); at the first
// rejection the next token is drawn from the positive residual max(p - q, 0),
// normalised; after every draft is accepted the bonus token is drawn from the
// target law of the bonus row.  The target law of row j is
//   p_j(v) = exp(x_j(v) / t - lse(x_j / t))   over the V unpadded lanes,
// t being the group's temperature.  The uniforms are inputs: u per draft row
// (accept iff u * q(d) < p(d)) and r per group (the draw: the smallest id v
// whose running sum of weights, in id order, exceeds r times the total).
//
// One CTA of 512 threads walks a group's chain, one row at a time (the rows
// of a group are dependent).  CTA b takes groups b, b + grid, ...  Per row:
//   pass 1  the row's temperature-scaled maximum and exp-sum (FP32, base 2:
//           a = x * log2(e) / t, L = log2 sum 2^a), 16-byte loads, each warp
//           over a contiguous range of the row;
//   accept  u * q(d) < 2^(a_d - L) with the draft's logit and q gathered;
//   draw    (first rejection, or the bonus row) pass 2 sums the weights in
//           FP64 per warp range (the residual max(p - q, 0) in FP32, or p);
//           the range holding r * total is split over the 512 threads, an
//           FP64 block scan of their sums finds the thread, and that thread
//           walks its few lanes.  A residual without mass (possible only
//           through rounding) falls back to p.
// Rows are read once for acceptance; the drawn row is read twice more (its
// weights need lse), plus one warp range of it.
#include <cuda_runtime.h>
#include <stdint.h>

#include "lp_internal.h"

namespace lp {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNegInf = -__builtin_huge_valf();
constexpr unsigned kStatusBadToken = 0x2u, kStatusBadGroup = 0x8u, kStatusBadTemperature = 0x20u;
constexpr int kChainThreads = 512;
constexpr int kChainWarps = kChainThreads / 32;
constexpr int kUnroll = 4;  // 16-byte loads in flight per lane in the row passes

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Eight consecutive lanes from an 8-aligned lane v0 < V.  Rows are 16-byte
// aligned and V_padded * element size is a multiple of 16, so a BF16 vector
// never leaves the row; an FP32 row may end after v0 + 4, and then the upper
// half is not loaded (those lanes lie past V and are never used).
template <int ELT>
__device__ __forceinline__ void load8(const void* row, long long v0, long long V, float (&x)[8]) {
    if constexpr (ELT == 2) {
        const uint4 w = __ldcs(reinterpret_cast<const uint4*>(reinterpret_cast<const unsigned short*>(row) + v0));
        const uint32_t a[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = __uint_as_float(a[i] << 16);
            x[2 * i + 1] = __uint_as_float(a[i] & 0xFFFF0000u);
        }
    } else {
        const float4* p = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(row) + v0);
        const float4 a = __ldcs(p);
        const float4 b = v0 + 4 < V ? __ldcs(p + 1) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    }
}

// The draft law's eight lanes from v0 (FP32 rows of the same stride).
__device__ __forceinline__ void loadq8(const float* q, long long v0, long long V, float (&y)[8]) {
    const float4* p = reinterpret_cast<const float4*>(q + v0);
    const float4 a = __ldcs(p);
    const float4 b = v0 + 4 < V ? __ldcs(p + 1) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    y[0] = a.x; y[1] = a.y; y[2] = a.z; y[3] = a.w;
    y[4] = b.x; y[5] = b.y; y[6] = b.z; y[7] = b.w;
}

template <int ELT>
__device__ __forceinline__ float logit(const void* row, long long v) {
    if constexpr (ELT == 2) {
        return __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short*>(row) + v) << 16);
    } else {
        return __ldg(reinterpret_cast<const float*>(row) + v);
    }
}

// Merges (m, s) pairs of sum 2^(a - m) (m = -inf: empty).
__device__ __forceinline__ void ms2_merge(float& m, float& s, float m2, float s2) {
    const float M = fmaxf(m, m2);
    if (M == kNegInf) return;
    s = (m > kNegInf ? s * ex2(m - M) : 0.0f) + (m2 > kNegInf ? s2 * ex2(m2 - M) : 0.0f);
    m = M;
}

struct ChainShared {
    float wm[kChainWarps], ws[kChainWarps];
    double wt[kChainWarps];      // weight total of each warp's range
    double tscan[kChainWarps];
    float L;                     // log2 sum 2^a of the current row
    int accept;                  // the current draft is accepted
    int range;                   // level 1: the warp range holding the target (-1: no weight)
    double before;               // level 1: the target less the weights before that range
    int first_th;                // level 2: first thread whose interval holds the target
    int last_th;                 // level 2: last thread with weight
    int token;                   // the drawn token
};

// Weight of lane v (value x, draft law q) in the current draw.
__device__ __forceinline__ float weight(float a, float L, float qv, bool residual) {
    const float pv = ex2(a - L);
    return residual ? fmaxf(pv - qv, 0.0f) : pv;
}

template <int ELT>
__global__ void __launch_bounds__(kChainThreads, 1) lp_chain_kernel(ChainParams p) {
    __shared__ ChainShared sm;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long V = p.V;
    // warp ranges: contiguous, 8-aligned
    const long long R = ((V + kChainWarps - 1) / kChainWarps + 7) & ~7ll;
    const long long w0 = (long long)warp * R, w1 = (w0 + R < V) ? w0 + R : V;
    for (int g = blockIdx.x; g < p.G; g += gridDim.x) {
        const int r0 = __ldg(&p.indptr[g]), r1 = __ldg(&p.indptr[g + 1]);
        const float t = __ldg(&p.temp[g]);
        const int k = r1 - r0 - 1;
        if (r0 < 0 || r1 > p.rows || k < 0 || k > p.k_max) {
            if (tid == 0) {
                atomicOr(p.status, kStatusBadGroup);
                p.accepted[g] = -1;
            }
            continue;
        }
        if (!(t > 0.0f) || !(t < __builtin_huge_valf())) {
            if (tid == 0) {
                atomicOr(p.status, kStatusBadTemperature);
                p.accepted[g] = -1;
            }
            for (int j = tid; j <= k; j += kChainThreads) p.emitted[r0 + j] = -1;
            continue;
        }
        const float scale = kLog2e / t;
        int a = 0;
        for (int j = 0; j <= k; ++j) {
            const long long row = (long long)r0 + j;
            const void* xr = reinterpret_cast<const unsigned char*>(p.logits) + row * p.Vp * ELT;
            // pass 1: max and exp-sum of a = x * scale over the row
            float m = kNegInf, s = 0.0f;
            for (long long vb = w0 + lane * 8; vb < w1; vb += kUnroll * 32 * 8) {
                float x[kUnroll][8];  // kUnroll loads in flight per lane
#pragma unroll
                for (int i = 0; i < kUnroll; ++i) {
                    const long long v0 = vb + (long long)i * 32 * 8;
                    if (v0 < w1) load8<ELT>(xr, v0, V, x[i]);
                }
#pragma unroll
                for (int i = 0; i < kUnroll; ++i) {
                    const long long v0 = vb + (long long)i * 32 * 8;
                    if (v0 >= w1) continue;
                    float vm = kNegInf;
#pragma unroll
                    for (int e = 0; e < 8; ++e) vm = (v0 + e < V) ? fmaxf(vm, x[i][e] * scale) : vm;
                    if (vm > m) {
                        s = (m > kNegInf) ? s * ex2(m - vm) : 0.0f;
                        m = vm;
                    }
#pragma unroll
                    for (int e = 0; e < 8; ++e) s += (v0 + e < V && m > kNegInf) ? ex2(x[i][e] * scale - m) : 0.0f;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ms2_merge(m, s, __shfl_xor_sync(kFull, m, o), __shfl_xor_sync(kFull, s, o));
            if (lane == 0) {
                sm.wm[warp] = m;
                sm.ws[warp] = s;
            }
            __syncthreads();
            if (tid == 0) {
                float M = sm.wm[0], S = sm.ws[0];
                for (int w = 1; w < kChainWarps; ++w) ms2_merge(M, S, sm.wm[w], sm.ws[w]);
                sm.L = M + lg2(S);
                if (p.lse_out) p.lse_out[row] = sm.L * kLn2;
            }
            __syncthreads();
            const float L = sm.L;
            const float* qr = p.q + row * p.Vp;
            bool residual = false;
            if (j < k) {
                // acceptance: u * q(d) < p(d)
                int accept = 0;
                if (tid == 0) {
                    const int d = __ldg(&p.drafts[row]);
                    if (d >= 0 && d < V) {
                        const float pd = ex2(logit<ELT>(xr, d) * scale - L);
                        accept = __ldg(&p.u[row]) * __ldg(&qr[d]) < pd;
                        if (accept) p.emitted[row] = d;
                    } else if (d >= V) {
                        atomicOr(p.status, kStatusBadToken);
                    }
                    sm.accept = accept;
                }
                __syncthreads();
                if (sm.accept) {
                    ++a;
                    __syncthreads();  // sm.accept is rewritten for the next row
                    continue;
                }
                residual = true;
            }
            // the draw: pass 2, FP64 weight totals of the warp ranges
            for (int attempt = 0; attempt < 2; ++attempt) {
                double acc = 0.0;
                for (long long vb = w0 + lane * 8; vb < w1; vb += kUnroll * 32 * 8) {
                    float x[kUnroll][8], qv[kUnroll][8];
#pragma unroll
                    for (int i = 0; i < kUnroll; ++i) {
                        const long long v0 = vb + (long long)i * 32 * 8;
                        if (v0 < w1) {
                            load8<ELT>(xr, v0, V, x[i]);
                            if (residual) loadq8(qr, v0, V, qv[i]);
                        }
                    }
#pragma unroll
                    for (int i = 0; i < kUnroll; ++i) {
                        const long long v0 = vb + (long long)i * 32 * 8;
                        if (v0 >= w1) continue;
                        float part = 0.0f;
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            part += (v0 + e < V) ? weight(x[i][e] * scale, L, residual ? qv[i][e] : 0.0f, residual)
                                                 : 0.0f;
                        acc += (double)part;
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(kFull, acc, o);
                if (lane == 0) sm.wt[warp] = acc;
                __syncthreads();
                if (tid == 0) {
                    // level 1: the first warp range whose running total exceeds r * total
                    double tot = 0.0;
                    for (int w = 0; w < kChainWarps; ++w) tot += sm.wt[w];
                    sm.range = -1;
                    if (tot > 0.0) {
                        const double target = (double)__ldg(&p.r[g]) * tot;
                        double run = 0.0, run_last = 0.0;
                        int last = -1;
                        for (int w = 0; w < kChainWarps; ++w) {
                            if (sm.wt[w] > 0.0) {
                                last = w;
                                run_last = run;
                                if (target < run + sm.wt[w]) {
                                    sm.range = w;
                                    break;
                                }
                            }
                            run += sm.wt[w];
                        }
                        if (sm.range < 0) sm.range = last;  // rounding put the target past the end
                        sm.before = sm.range == last ? run_last : run;
                        sm.before = target - sm.before;      // the target within the range
                    }
                }
                __syncthreads();
                if (sm.range >= 0) break;
                residual = false;  // a residual without mass (rounding): draw from p
                __syncthreads();
            }
            // level 2: the range split over the CTA's threads (contiguous sub-ranges)
            const int rw = sm.range;
            const double target = sm.before;
            const long long g0 = (long long)rw * R, g1 = (g0 + R < V) ? g0 + R : V;
            const long long per = (g1 - g0 + kChainThreads - 1) / kChainThreads;
            const long long s0 = g0 + (long long)tid * per, s1 = (s0 + per < g1) ? s0 + per : g1;
            double mine = 0.0;
            for (long long v = s0; v < s1; ++v)
                mine += (double)weight(logit<ELT>(xr, v) * scale, L, residual ? __ldg(&qr[v]) : 0.0f, residual);
            // block inclusive scan of the thread sums
            double incl = mine;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const double n = __shfl_up_sync(kFull, incl, o);
                if (lane >= o) incl += n;
            }
            if (lane == 31) sm.tscan[warp] = incl;
            if (tid == 0) {
                sm.first_th = 0x7FFFFFFF;
                sm.last_th = -1;
            }
            __syncthreads();
            if (warp == 0) {
                const double w = sm.tscan[lane];
                double wi = w;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const double n = __shfl_up_sync(kFull, wi, o);
                    if (lane >= o) wi += n;
                }
                sm.tscan[lane] = wi - w;  // exclusive prefix of the warps
            }
            __syncthreads();
            incl += sm.tscan[warp];
            const double excl = incl - mine;
            if (mine > 0.0) {
                if (target < incl) atomicMin(&sm.first_th, tid);
                atomicMax(&sm.last_th, tid);
            }
            __syncthreads();
            const int th = sm.first_th != 0x7FFFFFFF ? sm.first_th : sm.last_th;  // rounding: the last thread with weight
            if (tid == th) {
                double run = excl;
                int tok = -1, lastv = -1;
                for (long long v = s0; v < s1; ++v) {
                    const double w =
                        (double)weight(logit<ELT>(xr, v) * scale, L, residual ? __ldg(&qr[v]) : 0.0f, residual);
                    if (w > 0.0) {
                        lastv = (int)v;
                        run += w;
                        if (target < run) {
                            tok = (int)v;
                            break;
                        }
                    }
                }
                sm.token = tok >= 0 ? tok : lastv;
            }
            __syncthreads();
            if (tid == 0) {
                p.emitted[row] = sm.token;
                p.accepted[g] = a;
            }
            for (int jj = j + 1 + tid; jj <= k; jj += kChainThreads) p.emitted[r0 + jj] = -1;
            __syncthreads();
            break;
        }
    }
}

}  // namespace

cudaError_t launch_chain(const ChainParams& p, int dtype, int sms, cudaStream_t stream) {
    int grid = p.G < sms ? p.G : sms;
    if (grid < 1) grid = 1;
    if (dtype == 1) lp_chain_kernel<2><<<grid, kChainThreads, 0, stream>>>(p);
    else lp_chain_kernel<4><<<grid, kChainThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace lp
