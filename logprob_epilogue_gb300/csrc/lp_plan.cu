// lp_plan.cu -- host side of the C ABI (plan / bind / clip / run / score).
//
// The plan owns one device allocation holding the run's control block, work
// queue, per-row counters, group descriptors and per-tile partial results, sized
// once from the plan descriptor.  lp_run and lp_score only enqueue the three
// kernels (prepare, stream, records); nothing is allocated or synchronised on
// the hot path.
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>

#include "lp_epilogue.h"
#include "lp_internal.h"

struct lp_plan_s {
    lp_plan_desc d;
    int elt;
    int T;
    lp::LaunchCfg cfg;
    unsigned char* scratch;
    size_t scratch_bytes;
    lp::Ctrl* ctrl;
    unsigned long long* queue;
    unsigned int* tclaim;
    int* done;
    unsigned long long* row_best;
    int4* gdesc;
    ulonglong2* rec_tasks;
    ulonglong2* part_ms;
    int2* part_rank;
    unsigned long long* part_keys;
    size_t part_ms_bytes, part_keys_bytes;
    bool bound;
    lp_io io;
    const int32_t* clip_eos;     // lp_bind_clip inputs for lp_run (null: none)
    const int32_t* clip_budget;
    // optional host staging (LP_PLAN_HOST_STAGING)
    unsigned char* staging;
    size_t staging_bytes;
    lp_io stage_io;
    cudaStream_t last_stream;
    // optional vocabulary-shard exchange buffers (LP_PLAN_VOCAB_SHARDS)
    float2* shard_x1;   // [max_rows * kMaxShards]
    int* shard_x2;      // [max_rows * kMaxShards * 256]
    // optional timeline (LP_PLAN_DEBUG_TRACE)
    unsigned long long* trace;
    unsigned int* trace_count;
    int trace_cap, trace_ctas;
};

namespace {

thread_local int g_last_cuda_error = 0;

constexpr size_t kAlign = 256;
constexpr int64_t kDefaultTimeoutNs = 1000000000LL;  // 1 s

size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }

int cuda_fail(cudaError_t e) {
    g_last_cuda_error = (int)e;
    return LP_ECUDA;
}

int elt_of(int dtype) { return dtype == LP_BF16 ? 2 : (dtype == LP_F32 ? 4 : 0); }

int check_desc(const lp_plan_desc* d) {
    if (!d) return LP_EINVAL;
    if (elt_of(d->dtype) == 0) return LP_EDTYPE;
    if (d->max_rows < 1 || d->max_groups < 1 || d->V < 1 || d->V_padded < d->V) return LP_ESHAPE;
    if (d->V > (int64_t)0x7FFFFFFF - lp::tile_elems_of_dtype(d->dtype)) return LP_ESHAPE;
    if (d->k_max < 0 || d->k_max > LP_MAX_DRAFTS) return LP_ECAPACITY;
    if (d->k_alt_max < 0 || d->k_alt_max > LP_MAX_K_ALT) return LP_ECAPACITY;
    if (d->max_ids < 0 || d->max_ids > LP_MAX_IDS) return LP_ECAPACITY;
    if (d->max_groups > (1 << 26) || d->max_rows >= (1 << 28)) return LP_ECAPACITY;
    if ((d->V_padded * elt_of(d->dtype)) % 16 != 0) return LP_EALIGN;
    if (d->timeout_ns < 0) return LP_EINVAL;
    return LP_OK;
}

struct Layout {
    size_t ctrl, queue, tclaim, row_best, done, gdesc, rec_tasks, part_ms, part_rank, part_keys, total;
    size_t part_ms_bytes, part_keys_bytes;
};

Layout layout_of(const lp_plan_desc* d) {
    Layout L{};
    const size_t rows = (size_t)d->max_rows;
    const int64_t te = lp::tile_elems_of_dtype(d->dtype);
    const size_t T = (size_t)((d->V + te - 1) / te);
    size_t off = 0;
    L.ctrl = off;
    off = align_up(off + sizeof(lp::Ctrl));
    L.queue = off;
    off = align_up(off + rows * sizeof(unsigned long long));
    L.tclaim = off;
    off = align_up(off + rows * sizeof(unsigned int));
    L.row_best = off;
    off = align_up(off + rows * sizeof(unsigned long long));
    L.done = off;
    off = align_up(off + rows * sizeof(int));
    L.gdesc = off;
    off = align_up(off + (size_t)d->max_groups * sizeof(int4));
    L.rec_tasks = off;
    off = align_up(off + rows * 2 * sizeof(ulonglong2));
    L.part_ms = off;
    L.part_ms_bytes = rows * T * (lp::kConsumerThreads / 32) * sizeof(ulonglong2);
    off = align_up(off + L.part_ms_bytes);
    L.part_rank = off;
    off = align_up(off + rows * T * (lp::kConsumerThreads / 32) * sizeof(int2));
    L.part_keys = off;
    L.part_keys_bytes = rows * T * lp::kKeysPerTile * sizeof(unsigned long long);
    off = align_up(off + L.part_keys_bytes);
    L.total = off;
    return L;
}

struct StageLayout {
    size_t logits, indptr, drafts, sampled, requested, top_k, token_ids, id_counts;
    size_t records, accepted, emitted, lse, status, total;
};

StageLayout stage_layout_of(const lp_plan_desc* d) {
    StageLayout S{};
    const size_t rows = (size_t)d->max_rows, G = (size_t)d->max_groups;
    size_t off = 0;
    S.logits = off;
    off = align_up(off + rows * (size_t)d->V_padded * (size_t)elt_of(d->dtype));
    S.indptr = off;
    off = align_up(off + (G + 1) * 4);
    S.drafts = off;
    off = align_up(off + rows * 4);
    S.sampled = off;
    off = align_up(off + G * 4);
    S.requested = off;
    off = align_up(off + G * 4);
    S.top_k = off;
    off = align_up(off + G * 4);
    S.token_ids = off;
    off = align_up(off + G * LP_MAX_IDS * 4);
    S.id_counts = off;
    off = align_up(off + G * 4);
    S.records = off;
    off = align_up(off + rows * LP_RECORD_WORDS * 4);
    S.accepted = off;
    off = align_up(off + G * 4);
    S.emitted = off;
    off = align_up(off + rows * 4);
    S.lse = off;
    off = align_up(off + rows * 4);
    S.status = off;
    off = align_up(off + 4);
    S.total = off;
    return S;
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

int check_io(const lp_plan_s* plan, const lp_io* io) {
    if (!io) return LP_EINVAL;
    if (io->rows < 0 || io->groups < 0) return LP_ESHAPE;
    if (io->rows > plan->d.max_rows || io->groups > plan->d.max_groups) return LP_ESHAPE;
    if (!io->logits || !io->group_indptr || !io->draft_tokens || !io->sampled_tokens || !io->requested ||
        !io->top_k || !io->token_ids || !io->id_counts || !io->records || !io->accepted ||
        !io->emitted_tokens || !io->status)
        return LP_EINVAL;
    if (!aligned(io->logits, 16)) return LP_EALIGN;
    const void* i32s[] = {io->group_indptr, io->draft_tokens, io->sampled_tokens, io->requested, io->top_k,
                          io->token_ids,    io->id_counts,    io->records,        io->accepted,  io->emitted_tokens,
                          io->status};
    for (const void* q : i32s)
        if (!aligned(q, 4)) return LP_EALIGN;
    if (io->lse_out && !aligned(io->lse_out, 4)) return LP_EALIGN;
    return LP_OK;
}

lp::Params make_params(const lp_plan_s* plan, const lp_io& io) {
    lp::Params p{};
    p.logits = io.logits;
    p.V = plan->d.V;
    p.Vp = plan->d.V_padded;
    p.rows = io.rows;
    p.G = io.groups;
    p.T = plan->T;
    p.elt = plan->elt;
    p.k_max = plan->d.k_max;
    p.k_alt_max = plan->d.k_alt_max;
    p.max_ids = plan->d.max_ids;
    p.indptr = io.group_indptr;
    p.drafts = io.draft_tokens;
    p.sampled = io.sampled_tokens;
    p.requested = io.requested;
    p.top_k = io.top_k;
    p.token_ids = io.token_ids;
    p.id_counts = io.id_counts;
    p.records = io.records;
    p.accepted = io.accepted;
    p.emitted = io.emitted_tokens;
    p.lse_out = io.lse_out;
    p.status = io.status;
    p.ctrl = plan->ctrl;
    p.queue = plan->queue;
    p.tclaim = plan->tclaim;
    p.row_best = plan->row_best;
    p.done = plan->done;
    p.gdesc = plan->gdesc;
    p.rec_tasks = plan->rec_tasks;
    p.part_ms = plan->part_ms;
    p.part_rank = plan->part_rank;
    p.part_keys = plan->part_keys;
    p.timeout_ns = (unsigned long long)(plan->d.timeout_ns > 0 ? plan->d.timeout_ns : kDefaultTimeoutNs);
    p.debug_flags = plan->d.flags & LP_PLAN_DEBUG_FORCE_TIMEOUT;
    p.read_ahead = (plan->d.flags & LP_PLAN_READ_AHEAD) ? 1 : 0;
    p.done_last = p.T - 1 + (p.read_ahead ? lp::kParentDone : 0);
    p.trace = plan->trace;
    p.trace_count = plan->trace_count;
    p.trace_cap = plan->trace_cap;
    p.trace_ctas = plan->trace_ctas;
    return p;
}

// Makes the plan's device current for the scope; restores the caller's.
struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) {
            ok = false;
            return;
        }
        if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

}  // namespace

extern "C" {

size_t lp_plan_scratch_bytes(const lp_plan_desc* desc) {
    if (check_desc(desc) != LP_OK) return 0;
    size_t total = layout_of(desc).total;
    if (desc->flags & LP_PLAN_HOST_STAGING) total += stage_layout_of(desc).total;
    return total;
}

int lp_plan_create(lp_plan_t* out, const lp_plan_desc* desc) {
    if (!out) return LP_EINVAL;
    *out = nullptr;
    int rc = check_desc(desc);
    if (rc != LP_OK) return rc;
    DeviceGuard guard(desc->device);
    if (!guard.ok) return cuda_fail(cudaGetLastError());
    lp_plan_s* plan = new (std::nothrow) lp_plan_s();
    if (!plan) return LP_EINVAL;
    plan->d = *desc;
    plan->elt = elt_of(desc->dtype);
    plan->T = (int)((desc->V + lp::tile_elems_of_dtype(desc->dtype) - 1) / lp::tile_elems_of_dtype(desc->dtype));
    cudaError_t e = lp::query_launch_cfg(desc->dtype, &plan->cfg);
    if (e != cudaSuccess) {
        delete plan;
        return cuda_fail(e);
    }
    const Layout L = layout_of(desc);
    e = cudaMalloc(&plan->scratch, L.total);
    if (e != cudaSuccess) {
        delete plan;
        return cuda_fail(e);
    }
    plan->scratch_bytes = L.total;
    plan->ctrl = reinterpret_cast<lp::Ctrl*>(plan->scratch + L.ctrl);
    plan->queue = reinterpret_cast<unsigned long long*>(plan->scratch + L.queue);
    plan->tclaim = reinterpret_cast<unsigned int*>(plan->scratch + L.tclaim);
    plan->row_best = reinterpret_cast<unsigned long long*>(plan->scratch + L.row_best);
    plan->done = reinterpret_cast<int*>(plan->scratch + L.done);
    plan->gdesc = reinterpret_cast<int4*>(plan->scratch + L.gdesc);
    plan->rec_tasks = reinterpret_cast<ulonglong2*>(plan->scratch + L.rec_tasks);
    plan->part_ms = reinterpret_cast<ulonglong2*>(plan->scratch + L.part_ms);
    plan->part_rank = reinterpret_cast<int2*>(plan->scratch + L.part_rank);
    plan->part_keys = reinterpret_cast<unsigned long long*>(plan->scratch + L.part_keys);
    plan->part_ms_bytes = L.part_ms_bytes;
    plan->part_keys_bytes = L.part_keys_bytes;
    // all of it: the run epoch starts at 0, and no partial or record task then
    // carries the epoch of a run (never 0)
    e = cudaMemset(plan->scratch, 0, L.total);
    if (e == cudaSuccess && (desc->flags & LP_PLAN_HOST_STAGING)) {
        const StageLayout S = stage_layout_of(desc);
        e = cudaMalloc(&plan->staging, S.total);
        if (e == cudaSuccess) {
            plan->staging_bytes = S.total;
            lp_io& s = plan->stage_io;
            s.logits = plan->staging + S.logits;
            s.group_indptr = reinterpret_cast<const int32_t*>(plan->staging + S.indptr);
            s.draft_tokens = reinterpret_cast<const int32_t*>(plan->staging + S.drafts);
            s.sampled_tokens = reinterpret_cast<const int32_t*>(plan->staging + S.sampled);
            s.requested = reinterpret_cast<const int32_t*>(plan->staging + S.requested);
            s.top_k = reinterpret_cast<const int32_t*>(plan->staging + S.top_k);
            s.token_ids = reinterpret_cast<const int32_t*>(plan->staging + S.token_ids);
            s.id_counts = reinterpret_cast<const int32_t*>(plan->staging + S.id_counts);
            s.records = reinterpret_cast<int32_t*>(plan->staging + S.records);
            s.accepted = reinterpret_cast<int32_t*>(plan->staging + S.accepted);
            s.emitted_tokens = reinterpret_cast<int32_t*>(plan->staging + S.emitted);
            s.lse_out = reinterpret_cast<float*>(plan->staging + S.lse);
            s.status = reinterpret_cast<uint32_t*>(plan->staging + S.status);
        }
    }
    if (e == cudaSuccess && (desc->flags & LP_PLAN_VOCAB_SHARDS)) {
        const size_t rows = (size_t)desc->max_rows;
        e = cudaMalloc(&plan->shard_x1, rows * lp::kMaxShards * sizeof(float2));
        if (e == cudaSuccess) e = cudaMalloc(&plan->shard_x2, rows * lp::kMaxShards * lp::kShardWords * sizeof(int));
    }
    if (e == cudaSuccess && (desc->flags & LP_PLAN_DEBUG_TRACE)) {
        plan->trace_cap = 2048;
        plan->trace_ctas = plan->cfg.grid;
        const size_t ev = ((size_t)plan->trace_ctas * lp::kTraceRoles + 1) * plan->trace_cap * 2 * sizeof(unsigned long long);
        e = cudaMalloc(&plan->trace, ev);
        if (e == cudaSuccess) e = cudaMalloc(&plan->trace_count, (size_t)plan->trace_ctas * lp::kTraceRoles * sizeof(unsigned));
        if (e == cudaSuccess) e = cudaMemset(plan->trace, 0, ev);
        if (e == cudaSuccess) e = cudaMemset(plan->trace_count, 0, (size_t)plan->trace_ctas * lp::kTraceRoles * sizeof(unsigned));
    }
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        if (plan->trace) cudaFree(plan->trace);
        if (plan->trace_count) cudaFree(plan->trace_count);
        if (plan->shard_x1) cudaFree(plan->shard_x1);
        if (plan->shard_x2) cudaFree(plan->shard_x2);
        if (plan->staging) cudaFree(plan->staging);
        cudaFree(plan->scratch);
        delete plan;
        return cuda_fail(e);
    }
    *out = plan;
    return LP_OK;
}

int lp_plan_destroy(lp_plan_t plan) {
    if (!plan) return LP_EINVAL;
    DeviceGuard guard(plan->d.device);
    cudaError_t e = cudaSuccess;
    if (plan->trace) cudaFree(plan->trace);
    if (plan->trace_count) cudaFree(plan->trace_count);
    if (plan->shard_x1) cudaFree(plan->shard_x1);
    if (plan->shard_x2) cudaFree(plan->shard_x2);
    if (plan->staging) e = cudaFree(plan->staging);
    cudaError_t e2 = cudaFree(plan->scratch);
    delete plan;
    if (e != cudaSuccess) return cuda_fail(e);
    if (e2 != cudaSuccess) return cuda_fail(e2);
    return LP_OK;
}

int lp_bind(lp_plan_t plan, const lp_io* io) {
    if (!plan) return LP_EINVAL;
    const int rc = check_io(plan, io);
    if (rc != LP_OK) return rc;
    plan->io = *io;
    plan->bound = true;
    plan->clip_eos = nullptr;
    plan->clip_budget = nullptr;
    return LP_OK;
}

int lp_run_sharded(lp_plan_t plan, int32_t shards, void* stream) {
    if (!plan) return LP_EINVAL;
    if (!plan->bound || !plan->shard_x1) return LP_ESTATE;
    if (shards < 1 || shards > lp::kMaxShards || shards > plan->T) return LP_EINVAL;
    DeviceGuard guard(plan->d.device);
    if (!guard.ok) return cuda_fail(cudaGetLastError());
    lp::Params p = make_params(plan, plan->io);
    p.eos = plan->clip_eos;
    p.budget = plan->clip_budget;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = lp::launch_epilogue(p, plan->d.dtype, plan->cfg, s, false);
    if (e == cudaSuccess) e = lp::launch_shard_records(p, plan->d.dtype, plan->cfg, shards, plan->shard_x1,
                                                        plan->shard_x2, s);
    if (e != cudaSuccess) return cuda_fail(e);
    plan->last_stream = s;
    return LP_OK;
}

int lp_bind_clip(lp_plan_t plan, const int32_t* eos_tokens, const int32_t* budgets) {
    if (!plan) return LP_EINVAL;
    if (!plan->bound) return LP_ESTATE;
    if ((eos_tokens && !aligned(eos_tokens, 4)) || (budgets && !aligned(budgets, 4))) return LP_EALIGN;
    plan->clip_eos = eos_tokens;
    plan->clip_budget = budgets;
    return LP_OK;
}

int lp_run(lp_plan_t plan, void* stream) {
    if (!plan) return LP_EINVAL;
    if (!plan->bound) return LP_ESTATE;
    DeviceGuard guard(plan->d.device);
    if (!guard.ok) return cuda_fail(cudaGetLastError());
    lp::Params p = make_params(plan, plan->io);
    p.eos = plan->clip_eos;
    p.budget = plan->clip_budget;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const cudaError_t e = lp::launch_epilogue(p, plan->d.dtype, plan->cfg, s);
    if (e != cudaSuccess) return cuda_fail(e);
    plan->last_stream = s;
    return LP_OK;
}

namespace {
// The device address of a pinned host block mapped into the device's address
// space (16-byte aligned, as the tile copies need), or nullptr.
const void* mapped_host_logits(const void* h) {
    if (h == nullptr || (reinterpret_cast<uintptr_t>(h) & 15u) != 0) return nullptr;
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, h) != cudaSuccess) {
        cudaGetLastError();  // an unregistered pointer is not an error here
        return nullptr;
    }
    if (a.type != cudaMemoryTypeHost || a.devicePointer == nullptr) return nullptr;
    if ((reinterpret_cast<uintptr_t>(a.devicePointer) & 15u) != 0) return nullptr;
    return a.devicePointer;
}
}  // namespace

int lp_run_host_bytes(lp_plan_t plan, const lp_io* io, int64_t* h2d, int64_t* d2h) {
    if (!plan || !io || !h2d || !d2h) return LP_EINVAL;
    const int64_t rows = io->rows, G = io->groups;
    // mapped pinned logits are read in place (the rows the run reads, counted by the caller)
    const int64_t logit_bytes = mapped_host_logits(io->logits) ? 0 : rows * plan->d.V_padded * plan->elt;
    *h2d = logit_bytes + (G + 1) * 4 + rows * 4 + G * 4 * 4 + G * LP_MAX_IDS * 4 +
           rows * LP_RECORD_WORDS * 4 + G * 4 + rows * 4 + (io->lse_out ? rows * 4 : 0);
    *d2h = rows * LP_RECORD_WORDS * 4 + G * 4 + rows * 4 + (io->lse_out ? rows * 4 : 0) + 4;
    return LP_OK;
}

int lp_run_host(lp_plan_t plan, const lp_io* h, void* stream) {
    if (!plan) return LP_EINVAL;
    if (!plan->staging) return LP_ESTATE;
    int rc = check_io(plan, h);
    if (rc != LP_OK && rc != LP_EALIGN) return rc;  // host buffers need no device alignment
    DeviceGuard guard(plan->d.device);
    if (!guard.ok) return cuda_fail(cudaGetLastError());
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const lp_io& d = plan->stage_io;
    const size_t rows = (size_t)h->rows, G = (size_t)h->groups;
    const cudaMemcpyKind H2D = cudaMemcpyHostToDevice, D2H = cudaMemcpyDeviceToHost;
    struct Cp {
        void* dst;
        const void* src;
        size_t n;
        cudaMemcpyKind k;
    };
    // pinned, mapped logits are read in place: only the rows the run reads cross the link
    const void* mapped = mapped_host_logits(h->logits);
    const Cp in[] = {
        {(void*)d.logits, h->logits, mapped ? 0 : rows * (size_t)plan->d.V_padded * plan->elt, H2D},
        {(void*)d.group_indptr, h->group_indptr, (G + 1) * 4, H2D},
        {(void*)d.draft_tokens, h->draft_tokens, rows * 4, H2D},
        {(void*)d.sampled_tokens, h->sampled_tokens, G * 4, H2D},
        {(void*)d.requested, h->requested, G * 4, H2D},
        {(void*)d.top_k, h->top_k, G * 4, H2D},
        {(void*)d.token_ids, h->token_ids, G * LP_MAX_IDS * 4, H2D},
        {(void*)d.id_counts, h->id_counts, G * 4, H2D},
    };
    // outputs are staged in too, so rows the run does not write keep the caller's contents
    const Cp keep[] = {
        {d.records, h->records, rows * LP_RECORD_WORDS * 4, H2D},
        {d.accepted, h->accepted, G * 4, H2D},
        {d.emitted_tokens, h->emitted_tokens, rows * 4, H2D},
        {d.lse_out, h->lse_out, h->lse_out ? rows * 4 : 0, H2D},
    };
    for (const Cp& c : keep) {
        if (c.n == 0) continue;
        const cudaError_t e = cudaMemcpyAsync(c.dst, c.src, c.n, c.k, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    for (const Cp& c : in) {
        if (c.n == 0) continue;
        const cudaError_t e = cudaMemcpyAsync(c.dst, c.src, c.n, c.k, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    lp_io run_io = d;
    run_io.rows = h->rows;
    run_io.groups = h->groups;
    if (!h->lse_out) run_io.lse_out = nullptr;
    if (mapped) run_io.logits = mapped;
    lp::Params p = make_params(plan, run_io);
    p.host_logits = mapped ? 1 : 0;
    cudaError_t e = lp::launch_epilogue(p, plan->d.dtype, plan->cfg, s);
    if (e != cudaSuccess) return cuda_fail(e);
    const Cp out[] = {
        {h->records, d.records, rows * LP_RECORD_WORDS * 4, D2H},
        {h->accepted, d.accepted, G * 4, D2H},
        {h->emitted_tokens, d.emitted_tokens, rows * 4, D2H},
        {h->lse_out, d.lse_out, h->lse_out ? rows * 4 : 0, D2H},
        {h->status, d.status, 4, D2H},
    };
    for (const Cp& c : out) {
        if (c.n == 0) continue;
        e = cudaMemcpyAsync(c.dst, c.src, c.n, c.k, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    plan->last_stream = s;
    return LP_OK;
}

int lp_score(lp_plan_t plan, const lp_score_io* io, void* stream) {
    if (!plan || !io) return LP_EINVAL;
    if (io->rows < 0 || io->rows > plan->d.max_rows || io->rows > plan->d.max_groups) return LP_ESHAPE;
    if (io->rows > 0 && (!io->logits || !io->target_tokens || !io->records)) return LP_EINVAL;
    if (!io->status) return LP_EINVAL;
    if (!aligned(io->logits, 16)) return LP_EALIGN;
    if (!aligned(io->target_tokens, 4) || !aligned(io->records, 4) || !aligned(io->status, 4)) return LP_EALIGN;
    if (io->lse_out && !aligned(io->lse_out, 4)) return LP_EALIGN;
    DeviceGuard guard(plan->d.device);
    if (!guard.ok) return cuda_fail(cudaGetLastError());
    if (io->rows == 0) {  // nothing to score: status only
        const cudaError_t e0 = cudaMemsetAsync(io->status, 0, sizeof(uint32_t), static_cast<cudaStream_t>(stream));
        if (e0 != cudaSuccess) return cuda_fail(e0);
        plan->last_stream = static_cast<cudaStream_t>(stream);
        return LP_OK;
    }
    // the epilogue's machinery with one group per row (k = 0): no group vectors,
    // drafts or generation outputs
    lp_io g{};
    g.logits = io->logits;
    g.lse_out = io->lse_out;
    g.status = io->status;
    g.rows = io->rows;
    g.groups = io->rows;
    lp::Params p = make_params(plan, g);
    p.k_max = 0;
    p.targets = io->target_tokens;
    p.score_records = io->records;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const cudaError_t e = lp::launch_epilogue(p, plan->d.dtype, plan->cfg, s);
    if (e != cudaSuccess) return cuda_fail(e);
    plan->last_stream = s;
    return LP_OK;
}

int lp_chain_verify(lp_plan_t plan, const lp_chain_io* io, void* stream) {
    if (!plan || !io) return LP_EINVAL;
    if (io->rows < 0 || io->groups < 0) return LP_ESHAPE;
    if (io->rows > plan->d.max_rows || io->groups > plan->d.max_groups) return LP_ESHAPE;
    if (!io->status) return LP_EINVAL;
    if (io->groups > 0 && (!io->logits || !io->group_indptr || !io->draft_tokens || !io->draft_probs ||
                           !io->temperature || !io->u || !io->r || !io->accepted || !io->emitted))
        return LP_EINVAL;
    if (!aligned(io->logits, 16) || !aligned(io->draft_probs, 16)) return LP_EALIGN;
    const void* w4[] = {io->group_indptr, io->draft_tokens, io->temperature, io->u, io->r, io->accepted,
                        io->emitted, io->status};
    for (const void* q : w4)
        if (!aligned(q, 4)) return LP_EALIGN;
    if (io->lse_out && !aligned(io->lse_out, 4)) return LP_EALIGN;
    DeviceGuard guard(plan->d.device);
    if (!guard.ok) return cuda_fail(cudaGetLastError());
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(io->status, 0, sizeof(uint32_t), s);
    if (e == cudaSuccess && io->groups > 0) {
        lp::ChainParams c{};
        c.logits = io->logits;
        c.V = plan->d.V;
        c.Vp = plan->d.V_padded;
        c.rows = io->rows;
        c.G = io->groups;
        c.k_max = plan->d.k_max;
        c.indptr = io->group_indptr;
        c.drafts = io->draft_tokens;
        c.q = io->draft_probs;
        c.temp = io->temperature;
        c.u = io->u;
        c.r = io->r;
        c.accepted = io->accepted;
        c.emitted = io->emitted;
        c.lse_out = io->lse_out;
        c.status = io->status;
        e = lp::launch_chain(c, plan->d.dtype, plan->cfg.sms, s);
    }
    if (e != cudaSuccess) return cuda_fail(e);
    plan->last_stream = s;
    return LP_OK;
}

int lp_debug_tiles_read(lp_plan_t plan, int32_t* host_tiles, int32_t rows) {
    if (!plan || !host_tiles || rows < 0 || rows > plan->d.max_rows) return LP_EINVAL;
    DeviceGuard guard(plan->d.device);
    cudaError_t e = cudaStreamSynchronize(plan->last_stream);
    if (e == cudaSuccess && rows > 0) e = cudaMemcpy(host_tiles, plan->done, (size_t)rows * 4, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e);
    for (int32_t r = 0; r < rows; ++r) host_tiles[r] &= lp::kParentDone - 1;  // tile count only
    return LP_OK;
}

int lp_debug_poison_scratch(lp_plan_t plan, void* stream) {
    if (!plan) return LP_EINVAL;
    DeviceGuard guard(plan->d.device);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(plan->part_ms, 0xFF, plan->part_ms_bytes, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(plan->part_keys, 0xFF, plan->part_keys_bytes, s);
    // the scoring partials: one int2 per warp of a tile, half the size of part_ms
    if (e == cudaSuccess) e = cudaMemsetAsync(plan->part_rank, 0xFF, plan->part_ms_bytes / 2, s);
    // record tasks past the run's count are never read; all-ones words carry no run's epoch
    if (e == cudaSuccess)
        e = cudaMemsetAsync(plan->rec_tasks, 0xFF, (size_t)plan->d.max_rows * 2 * sizeof(ulonglong2), s);
    if (e != cudaSuccess) return cuda_fail(e);
    return LP_OK;
}

int lp_debug_occupy(int32_t device, int32_t ctas, int64_t ns, void* stream) {
    if (ctas < 1 || ns < 0 || ns > 10000000000LL) return LP_EINVAL;
    DeviceGuard guard(device);
    if (!guard.ok) return cuda_fail(cudaGetLastError());
    const cudaError_t e = lp::launch_occupy(ctas, (unsigned long long)ns, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? LP_OK : cuda_fail(e);
}

int lp_debug_trace(lp_plan_t plan, uint64_t* events, uint32_t* counts, int32_t* ctas, int32_t* cap) {
    if (!plan || !ctas || !cap) return LP_EINVAL;
    if (!plan->trace) return LP_ESTATE;
    *ctas = plan->trace_ctas;
    *cap = plan->trace_cap;
    if (!events) return LP_OK;
    if (!counts) return LP_EINVAL;
    DeviceGuard guard(plan->d.device);
    const size_t ev = ((size_t)plan->trace_ctas * lp::kTraceRoles + 1) * plan->trace_cap * 2 * sizeof(unsigned long long);
    cudaError_t e = cudaStreamSynchronize(plan->last_stream);
    if (e == cudaSuccess) e = cudaMemcpy(events, plan->trace, ev, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess)
        e = cudaMemcpy(counts, plan->trace_count, (size_t)plan->trace_ctas * lp::kTraceRoles * sizeof(unsigned),
                       cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e);
    return LP_OK;
}

int lp_plan_tiles_per_row(lp_plan_t plan) { return plan ? plan->T : LP_EINVAL; }

const char* lp_strerror(int code) {
    switch (code) {
        case LP_OK: return "ok";
        case LP_EINVAL: return "invalid argument (NULL pointer or nonsensical value)";
        case LP_ESHAPE: return "inconsistent sizes (V, V_padded, rows or groups beyond the plan)";
        case LP_EALIGN: return "misaligned buffer (logits need 16 bytes, int32 buffers 4; V_padded*elt multiple of 16)";
        case LP_ECAPACITY: return "request beyond the plan's limits (k_max, k_alt_max, max_ids)";
        case LP_EDTYPE: return "unknown dtype";
        case LP_ECUDA: return "CUDA runtime error (see lp_last_cuda_error)";
        case LP_ESTATE: return "plan not ready (nothing bound, or no host staging)";
        case LP_ESCRATCH: return "run needs more scratch than lp_run_static's fixed array (LP_STATIC_SCRATCH_BYTES)";
        default: return "unknown error code";
    }
}

int lp_last_cuda_error(void) { return g_last_cuda_error; }

}  // extern "C"

// ---------------------------------------------------------------- lp_run_static
//
// The same run as plan + bind + run, with its scratch in a fixed array of the
// library's device image instead of a cudaMalloc'd block (for callers that may
// not allocate device memory).  Every call shares the array.
namespace {

constexpr size_t kStaticScratchBytes = LP_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxStaticDevices = 64;
struct StaticDevice {
    bool ready;                 // device address looked up
    unsigned char* base;        // device address of g_static_scratch on this device
    bool cfg_ready[2];          // launch shape queried, per dtype
    lp::LaunchCfg cfg[2];
};
std::mutex g_static_mu;
StaticDevice g_static_dev[kMaxStaticDevices];

// One-time set-up of `dev` (current): the array's device address and the
// launch shape of `dtype`.  In host code g_static_scratch names a host-side
// shadow, so the kernels only ever get the address returned here.
cudaError_t static_setup(int dev, int dtype, unsigned char** base, lp::LaunchCfg* cfg) {
    std::lock_guard<std::mutex> lock(g_static_mu);
    StaticDevice& sd = g_static_dev[dev];
    if (!sd.ready) {
        void* ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_scratch);
        if (e != cudaSuccess) return e;
        if (ptr == nullptr) return cudaErrorInvalidSymbol;
        sd.base = static_cast<unsigned char*>(ptr);
        sd.ready = true;
    }
    if (!sd.cfg_ready[dtype]) {
        const cudaError_t e = lp::query_launch_cfg(dtype, &sd.cfg[dtype]);
        if (e != cudaSuccess) return e;
        sd.cfg_ready[dtype] = true;
    }
    *base = sd.base;
    *cfg = sd.cfg[dtype];
    return cudaSuccess;
}

}  // namespace

extern "C" int lp_run_static(const lp_plan_desc* desc, const lp_io* io, void* stream) {
    int rc = check_desc(desc);
    if (rc != LP_OK) return rc;
    if (desc->device < 0 || desc->device >= kMaxStaticDevices) return LP_EINVAL;
    // a plan object on the stack: never allocated, only carries the pointers
    lp_plan_s run{};
    run.d = *desc;
    run.d.flags &= ~(LP_PLAN_HOST_STAGING | LP_PLAN_DEBUG_TRACE);
    rc = check_io(&run, io);
    if (rc != LP_OK) return rc;
    // scratch sized for this run's rows and groups, not the descriptor's capacity
    lp_plan_desc need = run.d;
    need.max_rows = io->rows > 0 ? io->rows : 1;
    need.max_groups = io->groups > 0 ? io->groups : 1;
    const Layout L = layout_of(&need);
    if (L.total > kStaticScratchBytes) return LP_ESCRATCH;

    DeviceGuard guard(desc->device);
    if (!guard.ok) return cuda_fail(cudaGetLastError());
    unsigned char* base = nullptr;
    cudaError_t e = static_setup(desc->device, desc->dtype, &base, &run.cfg);
    if (e != cudaSuccess) return cuda_fail(e);
    run.elt = elt_of(desc->dtype);
    run.T = (int)((desc->V + lp::tile_elems_of_dtype(desc->dtype) - 1) / lp::tile_elems_of_dtype(desc->dtype));
    run.ctrl = reinterpret_cast<lp::Ctrl*>(base + L.ctrl);
    run.queue = reinterpret_cast<unsigned long long*>(base + L.queue);
    run.tclaim = reinterpret_cast<unsigned int*>(base + L.tclaim);
    run.row_best = reinterpret_cast<unsigned long long*>(base + L.row_best);
    run.done = reinterpret_cast<int*>(base + L.done);
    run.gdesc = reinterpret_cast<int4*>(base + L.gdesc);
    run.rec_tasks = reinterpret_cast<ulonglong2*>(base + L.rec_tasks);
    run.part_ms = reinterpret_cast<ulonglong2*>(base + L.part_ms);
    run.part_rank = reinterpret_cast<int2*>(base + L.part_rank);
    run.part_keys = reinterpret_cast<unsigned long long*>(base + L.part_keys);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The array keeps the previous call's contents.  The control block must
    // start at zero (its never-written word is the forced-timeout test's
    // flag), except the run epoch, which keeps counting across calls so that
    // no partial or record task left by an earlier call (at any layout) carries
    // the new run's epoch; the prepare kernel resets the queue, counters and
    // descriptors.
    e = cudaMemsetAsync(run.ctrl, 0, offsetof(lp::Ctrl, epoch), s);
    if (e != cudaSuccess) return cuda_fail(e);
    const lp::Params p = make_params(&run, *io);
    e = lp::launch_epilogue(p, desc->dtype, run.cfg, s);
    if (e != cudaSuccess) return cuda_fail(e);
    return LP_OK;
}
