// lp_oracle.cpp -- plain, slow CPU oracle for the logprob / greedy-acceptance
// epilogue.  TEST INFRASTRUCTURE ONLY: only the tests, the smoke check and the
// benchmark's CPU-baseline leg may load it.  It shares nothing with the CUDA
// library (no headers, helpers or constants).
//
// Every function follows the pages' definition step by step, with no blocking,
// fusion or reordering beyond what the definition states:
//   * "logprobs-design.md", generation-logprob contract: the logprob of a token
//     is its logit minus logsumexp over the full vocabulary, accumulated in
//     FP32 (here: the sum in FP64, rounded once to FP32, then an FP32
//     subtraction); alternatives ordered by decreasing logprob, then increasing
//     token id; up to 128 caller ids in caller order; the chosen token stored
//     separately; packed record = chosen id, chosen FP32 bits, then (id, bits)
//     pairs with -1 for unused ids; signed zero normalised; padded lanes never
//     enter; a zero request flag means no payload.
//   * "mtp-design.md", "A speculative round is a state transaction", steps 2-3:
//     verify rows [p, d0..d(K-1)]; with `a` accepted drafts the round emits a+1
//     tokens (a drafts and one target token).  Greedy acceptance compares each
//     draft with its row's argmax.
#include "lp_oracle.h"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <thread>
#include <vector>

namespace {

uint32_t float_bits(float f) {
    uint32_t u;
    std::memcpy(&u, &f, sizeof u);
    return u;
}

struct Pair {
    float lp;
    int32_t id;
};

}  // namespace

extern "C" float orc_lse(const float* x, int64_t V) {
    // Step 1: the maximum, to keep exp() in range (exact shift, any m works).
    double m = x[0];
    for (int64_t v = 1; v < V; ++v)
        if ((double)x[v] > m) m = x[v];
    // Step 2: sum of exp(x - m) over every unpadded lane, in double.
    double s = 0.0;
    for (int64_t v = 0; v < V; ++v) s += std::exp((double)x[v] - m);
    // Step 3: lse = m + log(s), rounded once to float (round to nearest even).
    double lse = m + std::log(s);
    return (float)lse;
}

extern "C" int32_t orc_argmax(const float* x, int64_t V) {
    // Strict '>' keeps the first (smallest) index among equal maxima; -0 and +0
    // compare equal under '>', so they are one value here.
    int32_t best = 0;
    for (int64_t v = 1; v < V; ++v)
        if (x[v] > x[best]) best = (int32_t)v;
    return best;
}

extern "C" float orc_logprob(float x, float lse) {
    volatile float d = x - lse;  // one FP32 subtraction, round to nearest
    float r = d;
    if (r == 0.0f) r = 0.0f;    // -0 -> +0
    return r;
}

extern "C" int32_t orc_topk(const float* x, int64_t V, float lse, int32_t K, int32_t* ids, float* lps) {
    std::vector<Pair> all((size_t)V);
    for (int64_t v = 0; v < V; ++v) all[(size_t)v] = Pair{orc_logprob(x[v], lse), (int32_t)v};
    // Built in ascending id order; a stable sort on "lp greater" keeps equal
    // values in ascending id order, which is the pages' tie rule.
    std::stable_sort(all.begin(), all.end(), [](const Pair& a, const Pair& b) { return a.lp > b.lp; });
    int32_t n = (int32_t)std::min<int64_t>(K, V);
    if (n < 0) n = 0;
    for (int32_t i = 0; i < n; ++i) {
        ids[i] = all[(size_t)i].id;
        lps[i] = all[(size_t)i].lp;
    }
    return n;
}

namespace {

struct Shared {
    const orc_io* io;
    std::atomic<int32_t> next_group{0};
    std::atomic<uint32_t> status{0};
    std::atomic<int64_t> rows_read{0};
};

void write_unused(int32_t* rec, int32_t from_pair) {
    for (int32_t i = from_pair; i < ORC_MAX_PAIRS; ++i) {
        rec[2 + 2 * i] = -1;
        rec[3 + 2 * i] = (int32_t)ORC_NAN_BITS;
    }
}

void run_group(Shared& sh, int32_t g) {
    const orc_io& io = *sh.io;
    const int32_t r0 = io.group_indptr[g];
    const int32_t k = io.group_indptr[g + 1] - r0 - 1;
    const bool flagged = io.requested[g] != 0;
    const int32_t sampled = io.sampled_tokens[g];
    uint32_t st = 0;

    // Request shape: a nonzero id count selects explicit ids, else K natural
    // alternatives.  Out-of-range values are clamped and flagged.
    int32_t count = io.id_counts[g];
    int32_t K = io.top_k[g];
    if (flagged) {
        if (count < 0 || count > io.max_ids) {
            st |= ORC_STATUS_BAD_COUNT;
            count = count < 0 ? 0 : io.max_ids;
        }
        if (count == 0 && (K < 0 || K > io.k_alt_max)) {
            st |= ORC_STATUS_BAD_COUNT;
            K = K < 0 ? 0 : io.k_alt_max;
        }
    }

    // Commit clipping ("mtp-design.md", a speculative round, step 4): the
    // emitted prefix of length t (1 <= t <= a+1) ends at the first emitted EOS
    // token (which is emitted) and holds at most `budget` tokens.  A request
    // already at its limit (budget <= 0) takes no step: nothing is emitted,
    // read or written, and accepted is -1.
    const int32_t eos = io.eos_tokens ? io.eos_tokens[g] : -1;
    const int32_t budget = io.budgets ? io.budgets[g] : INT32_MAX;
    if (budget <= 0) {
        io.accepted[g] = -1;
        for (int32_t j = 0; j <= k; ++j) io.emitted_tokens[(int64_t)r0 + j] = -1;
        sh.status.fetch_or(st);
        return;
    }

    // A k=0 request with a caller-sampled token and no flag needs no logits.
    const bool must_read = flagged || k >= 1 || sampled < 0;
    if (!must_read) {
        if (sampled >= io.V) st |= ORC_STATUS_BAD_TOKEN;
        io.emitted_tokens[r0] = sampled;
        io.accepted[g] = 0;
        sh.status.fetch_or(st);
        return;
    }

    int64_t read = 0;
    for (int32_t j = 0; j <= k; ++j) {
        const int64_t row = (int64_t)r0 + j;
        const float* x = io.logits + row * io.Vp;
        const int32_t amax = orc_argmax(x, io.V);
        ++read;
        int32_t chosen = amax;
        if (k == 0 && sampled >= 0) {
            chosen = sampled;
            if (sampled >= io.V) st |= ORC_STATUS_BAD_TOKEN;
        }
        io.emitted_tokens[row] = chosen;

        if (flagged) {
            const float lse = orc_lse(x, io.V);
            if (io.lse_out) io.lse_out[row] = lse;
            int32_t* rec = io.records + row * ORC_RECORD_WORDS;
            rec[0] = chosen;
            rec[1] = (chosen >= 0 && chosen < io.V) ? (int32_t)float_bits(orc_logprob(x[chosen], lse))
                                                    : (int32_t)ORC_NAN_BITS;
            int32_t used = 0;
            if (count > 0) {
                const int32_t* tid = io.token_ids + (int64_t)g * ORC_MAX_PAIRS;
                for (int32_t i = 0; i < count; ++i) {
                    const int32_t id = tid[i];
                    rec[2 + 2 * i] = id;
                    if (id >= 0 && id < io.V) {
                        rec[3 + 2 * i] = (int32_t)float_bits(orc_logprob(x[id], lse));
                    } else {
                        rec[3 + 2 * i] = (int32_t)ORC_NAN_BITS;
                        st |= ORC_STATUS_BAD_ID;
                    }
                }
                used = count;
            } else if (K > 0) {
                std::vector<int32_t> ids((size_t)K);
                std::vector<float> lps((size_t)K);
                used = orc_topk(x, io.V, lse, K, ids.data(), lps.data());
                for (int32_t i = 0; i < used; ++i) {
                    rec[2 + 2 * i] = ids[(size_t)i];
                    rec[3 + 2 * i] = (int32_t)float_bits(lps[(size_t)i]);
                }
            }
            write_unused(rec, used);
        }

        // Row j < k accepts its draft when the draft equals the row's argmax;
        // the first mismatch (or the bonus row j == k) ends the group.  The
        // clip ends it too, at an emitted EOS or once `budget` tokens are
        // emitted, so t = min(a + 1, budget, position of the first EOS + 1)
        // and no row past the clipped prefix is read.
        const bool accept = j < k && io.draft_tokens[row] == amax;
        const bool clipped = (eos >= 0 && chosen == eos) || j + 1 >= budget;
        if (!accept || clipped) {
            io.accepted[g] = j;
            for (int32_t jj = j + 1; jj <= k; ++jj) io.emitted_tokens[(int64_t)r0 + jj] = -1;
            break;
        }
    }
    sh.rows_read.fetch_add(read);
    sh.status.fetch_or(st);
}

bool groups_valid(const orc_io& io) {
    if (io.groups < 0) return false;
    if (io.groups == 0) return true;
    if (io.group_indptr[0] < 0 || io.group_indptr[io.groups] > io.rows) return false;
    for (int32_t g = 0; g < io.groups; ++g) {
        const int32_t size = io.group_indptr[g + 1] - io.group_indptr[g];
        if (size < 1 || size - 1 > io.k_max) return false;
    }
    return true;
}

}  // namespace

extern "C" int orc_epilogue(const orc_io* io, int threads) {
    if (!io || !io->logits || !io->group_indptr || !io->draft_tokens || !io->sampled_tokens ||
        !io->requested || !io->top_k || !io->token_ids || !io->id_counts || !io->records ||
        !io->accepted || !io->emitted_tokens || !io->status)
        return -1;
    if (!groups_valid(*io)) {
        // Malformed group layout: nothing is read or written.
        *io->status = ORC_STATUS_BAD_GROUP;
        if (io->rows_read) *io->rows_read = 0;
        return 0;
    }
    Shared sh;
    sh.io = io;
    auto worker = [&sh]() {
        for (;;) {
            const int32_t g = sh.next_group.fetch_add(1);
            if (g >= sh.io->groups) break;
            run_group(sh, g);
        }
    };
    if (threads <= 1) {
        worker();
    } else {
        std::vector<std::thread> pool;
        for (int t = 0; t < threads; ++t) pool.emplace_back(worker);
        for (auto& th : pool) th.join();
    }
    *io->status = sh.status.load();
    if (io->rows_read) *io->rows_read = sh.rows_read.load();
    return 0;
}

// ---- prompt scoring ("logprobs-design.md", the prompt-logprobs paragraphs:
// each scored row holds the actual token id, its raw FP32 logprob bits, its
// rank, then twenty (id, logprob bits) alternatives in the generation order;
// an invalid target row holds id -1, NaN, rank zero and alternative ids -1).

extern "C" int32_t orc_rank(const float* x, int64_t V, float lse, float lp) {
    // The definition: one plus the number of lanes whose reported value
    // fl32(x_v - lse) is strictly greater than the target's.
    int32_t greater = 0;
    for (int64_t v = 0; v < V; ++v)
        if (orc_logprob(x[v], lse) > lp) ++greater;
    return 1 + greater;
}

namespace {

void score_row(const float* x, int64_t V, int32_t t, int32_t* rec, float* lse_out, uint32_t* st) {
    if (t < 0 || t >= V) {
        if (t >= V) *st |= ORC_STATUS_BAD_TOKEN;
        rec[0] = -1;
        rec[1] = (int32_t)ORC_NAN_BITS;
        rec[2] = 0;
        for (int32_t i = 0; i < ORC_SCORE_ALTS; ++i) {
            rec[3 + 2 * i] = -1;
            rec[4 + 2 * i] = (int32_t)ORC_NAN_BITS;
        }
        return;
    }
    const float lse = orc_lse(x, V);
    if (lse_out) *lse_out = lse;
    const float lp = orc_logprob(x[t], lse);
    rec[0] = t;
    rec[1] = (int32_t)float_bits(lp);
    rec[2] = orc_rank(x, V, lse, lp);
    int32_t ids[ORC_SCORE_ALTS];
    float lps[ORC_SCORE_ALTS];
    const int32_t n = orc_topk(x, V, lse, ORC_SCORE_ALTS, ids, lps);
    for (int32_t i = 0; i < ORC_SCORE_ALTS; ++i) {
        rec[3 + 2 * i] = i < n ? ids[i] : -1;
        rec[4 + 2 * i] = i < n ? (int32_t)float_bits(lps[i]) : (int32_t)ORC_NAN_BITS;
    }
}

}  // namespace

extern "C" int orc_score(const float* logits, int64_t rows, int64_t V, int64_t Vp, const int32_t* targets,
                         int32_t* records, float* lse_out, uint32_t* status, int threads) {
    if (!logits || !targets || !records || !status) return -1;
    std::atomic<int64_t> next{0};
    std::atomic<uint32_t> st_all{0};
    auto worker = [&]() {
        for (;;) {
            const int64_t r = next.fetch_add(1);
            if (r >= rows) break;
            uint32_t st = 0;
            score_row(logits + r * Vp, V, targets[r], records + r * ORC_SCORE_WORDS, lse_out ? lse_out + r : nullptr,
                      &st);
            st_all.fetch_or(st);
        }
    };
    if (threads <= 1) {
        worker();
    } else {
        std::vector<std::thread> pool;
        for (int t = 0; t < threads; ++t) pool.emplace_back(worker);
        for (auto& th : pool) th.join();
    }
    *status = st_all.load();
    return 0;
}

// ---- stochastic chain verification ("mtp-design.md", "Sampling correctness":
// accept with probability min(1, p/q), on rejection draw the normalised
// positive residual, after full acceptance draw the bonus from the target law).

namespace {

// Target law of one row at temperature t: p(v) = exp(x_v/t - lse(x/t)), FP64.
void target_law(const float* x, int64_t V, double t, std::vector<double>& p) {
    p.assign((size_t)V, 0.0);
    double m = -INFINITY;
    for (int64_t v = 0; v < V; ++v) m = std::max(m, (double)x[v] / t);
    double s = 0.0;
    for (int64_t v = 0; v < V; ++v) s += std::exp((double)x[v] / t - m);
    const double log_z = m + std::log(s);  // log of the normaliser
    for (int64_t v = 0; v < V; ++v) p[(size_t)v] = std::exp((double)x[v] / t - log_z);
}

// Inverse CDF over ids in ascending order: the smallest v whose running sum of
// w exceeds r * sum(w).  Zero-weight lanes are never drawn.
int32_t draw(const std::vector<double>& w, double r) {
    double total = 0.0;
    for (double x : w) total += x;
    const double target = r * total;
    double c = 0.0;
    int32_t last = -1;
    for (size_t v = 0; v < w.size(); ++v) {
        if (w[v] <= 0.0) continue;
        c += w[v];
        last = (int32_t)v;
        if (c > target) return (int32_t)v;
    }
    return last;  // rounding left the target at the total: the last lane with mass
}

}  // namespace

extern "C" int orc_chain_verify(const float* logits, int64_t rows, int64_t V, int64_t Vp, int32_t groups,
                                const int32_t* group_indptr, const int32_t* draft_tokens,
                                const float* draft_probs, const float* temperature, const float* u,
                                const float* r, int32_t* accepted, int32_t* emitted) {
    if (!logits || !group_indptr || !draft_tokens || !draft_probs || !temperature || !u || !r || !accepted ||
        !emitted)
        return -1;
    (void)rows;
    std::vector<double> p, w;
    for (int32_t g = 0; g < groups; ++g) {
        const double t = temperature[g];
        if (!(t > 0.0)) return -1;
        const int32_t r0 = group_indptr[g];
        const int32_t k = group_indptr[g + 1] - r0 - 1;
        int32_t a = 0;
        int32_t last = -1;
        for (int32_t j = 0; j <= k; ++j) {
            const int64_t row = (int64_t)r0 + j;
            target_law(logits + row * Vp, V, t, p);
            if (j == k) {  // every draft accepted: the bonus token from the target law
                last = draw(p, (double)r[g]);
                break;
            }
            const int32_t d = draft_tokens[row];
            const float* q = draft_probs + row * Vp;
            const double pd = (d >= 0 && d < V) ? p[(size_t)d] : 0.0;
            const double qd = (d >= 0 && d < V) ? (double)q[d] : 0.0;
            if ((double)u[row] * qd < pd) {  // u < p/q: draft j accepted
                emitted[row] = d;
                ++a;
                continue;
            }
            // the first rejection: draw from max(p - q, 0), normalised
            w.assign((size_t)V, 0.0);
            double mass = 0.0;
            for (int64_t v = 0; v < V; ++v) {
                w[(size_t)v] = std::max(p[(size_t)v] - (double)q[v], 0.0);
                mass += w[(size_t)v];
            }
            last = draw(mass > 0.0 ? w : p, (double)r[g]);
            break;
        }
        accepted[g] = a;
        emitted[(int64_t)r0 + a] = last;
        for (int32_t j = a + 1; j <= k; ++j) emitted[(int64_t)r0 + j] = -1;
    }
    return 0;
}
