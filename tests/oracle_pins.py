"""Pins for the CPU oracle: checks against what the pages and mathematics fix.

Each pin is a function of an oracle handle (``oracle.load()`` or a mutated
copy), so the same pins can show that a planted mistake is caught.  Sources:

  * "logprobs-design.md", generation-logprob contract: lp = logit - logsumexp
    over the full vocabulary (FP32), alternatives by decreasing logprob then
    increasing id, signed zero normalised, padded lanes excluded, explicit ids
    in caller order, packed record with -1 for unused ids.
  * "mtp-design.md", "A speculative round is a state transaction", steps 2-3:
    a accepted drafts => a+1 emitted tokens.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "oracle_cases.json")
NAN_BITS = 0x7FC00000


def _num(v) -> np.float32:
    return np.float32(float(v))  # "-0.0" strings keep the sign


def _golden_row(case) -> np.ndarray:
    if "x" in case:
        return np.array([_num(v) for v in case["x"]], np.float32)
    spec = case["x_spec"]
    x = np.full(spec["V"], np.float32(spec["fill"]), np.float32)
    for lo, hi, val in spec["set"]:
        x[lo:hi + 1] = np.float32(val)
    return x


def f32_ulp(v: np.float32) -> float:
    v = np.float32(v)
    return float(np.spacing(np.abs(v)))


def bits(v) -> int:
    return int(np.array([v], np.float32).view(np.uint32)[0])


def brute_force_order(lp: np.ndarray) -> np.ndarray:
    """O(V^2) rank count: rank(v) = #{u: lp_u > lp_v or (lp_u == lp_v and u < v)}."""
    V = lp.shape[0]
    ranks = np.empty(V, np.int64)
    for v in range(V):
        gt = np.count_nonzero(lp > lp[v])
        eq_before = np.count_nonzero(lp[:v] == lp[v])
        ranks[v] = gt + eq_before
    order = np.empty(V, np.int64)
    order[ranks] = np.arange(V)
    return order


def independent_lse(x: np.ndarray) -> np.float32:
    """math.fsum-based logsumexp in double (a different summation than the oracle's)."""
    xs = [float(v) for v in x]
    m = max(xs)
    return np.float32(m + math.log(math.fsum(math.exp(v - m) for v in xs)))


# ----------------------------------------------------------------------------- pins

def pin_golden_rows(orc):
    cases = json.load(open(GOLDEN))["rows"]
    for c in cases:
        x = _golden_row(c)
        want_lse = np.float32(eval(c["lse_expr"], {"math": math}))
        got_lse = orc.lse(x)
        assert abs(float(got_lse) - float(want_lse)) <= f32_ulp(want_lse), (c["name"], got_lse, want_lse)
        assert bits(got_lse) == bits(want_lse) or c["name"] not in ("subtraction_induced_ties", "single_lane_negative_zero"), c["name"]
        ids, lps = orc.topk(x, c["K"])
        assert ids.tolist() == c["expected_ids"], (c["name"], ids.tolist())
        for sid, b in c.get("expected_lp_bits", {}).items():
            pos = ids.tolist().index(int(sid))
            assert bits(lps[pos]) == b, (c["name"], sid, hex(bits(lps[pos])), hex(b))
        assert orc.argmax(x) == c["expected_argmax"], c["name"]
        # every reported lp is fl32(x - lse) computed here with numpy float32
        for i, v in zip(ids, lps):
            want = np.float32(x[i]) - np.float32(got_lse)
            want = np.float32(0.0) if want == 0 else want
            assert bits(v) == bits(want), (c["name"], int(i))


def pin_golden_groups(orc):
    for c in json.load(open(GOLDEN))["groups"]:
        V = c["V"]
        rows = np.array([[_num(v) for v in r] for r in c["rows"]], np.float32)
        n = rows.shape[0]
        w = W.custom(rows, V, [n], drafts=c["drafts"], top_k=[2], k_max=n - 1)
        sentinel = np.full((n, 258), 0x5A5A5A5A, np.int32)
        r = orc.epilogue(w.logits_f32(), V, **w.inputs(), k_max=w.k_max, records=sentinel.copy())
        for j, a in enumerate(c["expected_argmax"]):
            assert orc.argmax(rows[j]) == a, (c["name"], j)
        assert int(r["accepted"][0]) == c["expected_accepted"], c["name"]
        assert r["emitted_tokens"].tolist() == c["expected_emitted"], c["name"]
        assert r["rows_read"] == c["expected_rows_read"], c["name"]
        acc = c["expected_accepted"]
        for j in range(n):
            if j <= acc:
                assert r["records"][j, 0] == c["expected_emitted"][j]
                assert r["records"][j, 2 + 2 * 2] == -1 and r["records"][j, 3 + 2 * 2] == NAN_BITS
            else:
                assert (r["records"][j] == 0x5A5A5A5A).all(), (c["name"], j)


def _bf_rows(rng):
    out = []
    for V in (1, 2, 3, 5, 17, 33, 64, 100):
        out.append(("random", rng.normal(0, 3, V).astype(np.float32)))
        out.append(("tied", np.round(rng.normal(0, 1, V) * 2).astype(np.float32) / 2))
        z = rng.normal(0, 1, V).astype(np.float32)
        m = rng.random(V) < 0.4
        z[m] = np.where(rng.random(m.sum()) < 0.5, np.float32(-0.0), np.float32(0.0))
        out.append(("signed_zero", z))
    # a row whose subtraction merges distinct logits
    out.append(("collapse", np.concatenate([[np.float32(3000.0)], rng.uniform(0, 0.01, 60).astype(np.float32)])))
    return out


def pin_brute_force(orc):
    rng = np.random.default_rng(1234)
    for kind, x in _bf_rows(rng):
        lse = orc.lse(x)
        lp = (x.astype(np.float32) - np.float32(lse)).astype(np.float32)
        lp[lp == 0] = np.float32(0.0)
        order = brute_force_order(lp)
        am = int(np.flatnonzero(x == x.max())[0])
        assert orc.argmax(x) == am, kind
        for K in (0, 1, 5, 20, 25):
            ids, lps = orc.topk(x, K, lse)
            n = min(K, x.size)
            assert ids.tolist() == order[:n].tolist(), (kind, x.size, K)
            assert [bits(v) for v in lps] == [bits(lp[i]) for i in order[:n]], (kind, x.size, K)


def pin_lse_independent(orc):
    import torch
    rng = np.random.default_rng(99)
    cases = [rng.normal(0, s, V).astype(np.float32) for s, V in ((1, 7), (3, 1000), (3, 248_320), (4, 20_000))]
    cases.append(np.full(513, np.float32(-7.25), np.float32))
    for x in cases:
        got = orc.lse(x)
        a = independent_lse(x)
        b = np.float32((torch.from_numpy(x.astype(np.float64))[0]
                        - torch.log_softmax(torch.from_numpy(x.astype(np.float64)), 0)[0]).item())
        for want in (a, b):
            assert abs(float(got) - float(want)) <= f32_ulp(want), (x.size, got, want)


def pin_two_value_closed_form(orc):
    for a, d in ((0.0, 0.5), (10.0, 3.0), (-4.0, 20.0), (1e3, 1e-3)):
        x = np.array([a, a - d], np.float32)
        want = np.float32(float(x[0]) + math.log1p(math.exp(float(x[1]) - float(x[0]))))
        got = orc.lse(x)
        assert abs(float(got) - float(want)) <= f32_ulp(want), (a, d, got, want)
        lp0 = orc.logprob(x[0], got)
        assert bits(lp0) == bits(np.float32(x[0]) - got), (a, d)


def pin_sum_exp_invariant(orc):
    rng = np.random.default_rng(5)
    for V, s in ((1000, 2.0), (151_936, 2.5), (262_144, 4.0)):
        x = rng.normal(0, s, V).astype(np.float32)
        lse = orc.lse(x)
        total = float(np.exp(x.astype(np.float64) - np.float64(lse)).sum())
        assert abs(total - 1.0) <= 1e-5, (V, total)


def pin_pad_exclusion(orc):
    w = W.tiny()
    base = orc.epilogue(w.logits_f32(), w.V, **w.inputs(), k_max=w.k_max)
    x = w.logits_f32().copy()
    x[:, w.V:] = np.float32(-3.0)        # different pad contents
    alt = orc.epilogue(x, w.V, **w.inputs(), k_max=w.k_max)
    for key in ("records", "accepted", "emitted_tokens"):
        assert np.array_equal(base[key], alt[key]), key
    # and a leak of +1e30 pads would make lse ~1e30
    assert np.nanmax(base["lse"]) < 100.0


def pin_id_passthrough(orc):
    rng = np.random.default_rng(7)
    x = rng.normal(0, 2, 300).astype(np.float32)
    ids = [299, 0, 17, 5, 128, 64]
    lse = orc.lse(x)
    nat_ids, nat_lps = orc.topk(x, 300, lse)
    nat = {int(i): bits(v) for i, v in zip(nat_ids, nat_lps)}
    w = W.custom(x[None, :], 300, [1], top_k=[20], token_ids=[ids], id_counts=[len(ids)])
    r = orc.epilogue(w.logits_f32(), 300, **w.inputs())
    rec = r["records"][0]
    for i, tid in enumerate(ids):
        assert rec[2 + 2 * i] == tid
        assert (int(rec[3 + 2 * i]) & 0xFFFFFFFF) == nat[tid]
    for i in range(len(ids), 128):
        assert rec[2 + 2 * i] == -1 and rec[3 + 2 * i] == NAN_BITS


def pin_acceptance_prefixes(orc):
    rng = np.random.default_rng(11)
    k, V = 5, 64
    for a in range(k + 1):
        rows = rng.normal(0, 1, (k + 1, V)).astype(np.float32)
        am = rng.integers(0, V, k + 1)
        rows[np.arange(k + 1), am] = 10.0
        drafts = np.full(k + 1, -1, np.int32)
        drafts[:k] = am[:k]
        if a < k:
            drafts[a] = (am[a] + 1) % V
        w = W.custom(rows, V, [k + 1], drafts=drafts, top_k=[3], k_max=k)
        sentinel = np.full((k + 1, 258), 0x33, np.int32)
        r = orc.epilogue(w.logits_f32(), V, **w.inputs(), k_max=k, records=sentinel.copy())
        assert int(r["accepted"][0]) == a
        assert r["rows_read"] == a + 1
        want = [int(am[j]) for j in range(a + 1)] + [-1] * (k - a)
        assert r["emitted_tokens"].tolist() == want, (a, r["emitted_tokens"])
        for j in range(k + 1):
            if j <= a:
                assert r["records"][j, 0] == am[j] and r["records"][j, 2] == am[j]
            else:
                assert (r["records"][j] == 0x33).all()


def pin_tiny_workload(orc):
    w = W.tiny()
    sentinel = np.full((w.rows, 258), 0x11, np.int32)
    r = orc.epilogue(w.logits_f32(), w.V, **w.inputs(), k_max=w.k_max, records=sentinel.copy())
    assert r["accepted"].tolist() == [2, 0, 0]
    assert r["rows_read"] == 4                      # rows 0, 1, 2 and 4
    em = r["emitted_tokens"].tolist()
    assert em[:3] == [int(w.draft_tokens[0]), int(w.draft_tokens[1]), int(w.planted_argmax[2])]
    assert em[3] == -1 and em[4] == int(w.sampled_tokens[1]) and em[5] == int(w.sampled_tokens[2])
    assert (r["records"][3] == 0x11).all() and (r["records"][5] == 0x11).all()
    rec4 = r["records"][4]
    assert [int(rec4[2 + 2 * i]) for i in range(15)] == w.token_ids[1, :15].tolist()
    assert w.token_ids[1, :3].tolist() == [7, 999, 3]
    assert r["status"] == 0


def pin_wide_tie(orc):
    w = W.wide()
    r = orc.epilogue(w.logits_f32(), w.V, **w.inputs(), k_max=w.k_max)
    assert r["accepted"].tolist() == [3]
    x = w.logits_f32(3)
    tied = np.flatnonzero(x[:w.V] == np.float32(16.0))
    assert tied.size == 64
    rec = r["records"][3]
    assert [int(rec[2 + 2 * i]) for i in range(20)] == sorted(tied.tolist())[:20]
    assert rec[0] == tied.min()


def pin_status_bits(orc):
    x = np.arange(10, dtype=np.float32)[None, :].repeat(3, 0)
    # bad explicit id, bad sampled token, bad count
    w = W.custom(x, 10, [1, 1, 1], sampled=[-1, 12, -1], requested=[1, 0, 1], top_k=[20, 0, 40],
                 token_ids=[[3, 10, -2], None, None], id_counts=[3, 0, 0])
    r = orc.epilogue(w.logits_f32(), 10, **w.inputs())
    rec = r["records"][0]
    assert rec[2:8].view(np.uint32).tolist() == [3, bits(np.float32(3) - orc.lse(x[0])), 10, NAN_BITS,
                                                 0xFFFFFFFE, NAN_BITS]
    assert r["status"] == (0x1 | 0x2 | 0x4)
    assert r["emitted_tokens"][1] == 12
    assert r["rows_read"] == 2          # row 1: unflagged k=0 with a sampled token is not read
    # malformed groups: nothing written
    w2 = W.custom(x, 10, [2, 1], k_max=0)
    r2 = orc.epilogue(w2.logits_f32(), 10, **w2.inputs(), k_max=0)
    assert r2["status"] == 0x8 and r2["rows_read"] == 0
    assert (r2["emitted_tokens"] == -7).all()


# ----------------------------------------------------------------------------- prompt scoring
#
# "logprobs-design.md", the prompt-logprobs paragraphs: a scored row holds the
# actual token id, its FP32 logprob bits, its rank (one plus the count of
# strictly greater reported values), then twenty alternatives in the generation
# order; an invalid target row holds id -1, NaN, rank zero and alternative ids -1.

SCORE_WORDS = 43


def u32(v) -> int:
    return int(v) & 0xFFFFFFFF


def _score_rows(rng):
    yield rng.normal(0, 2, 500).astype(np.float32)
    yield (np.round(rng.normal(0, 2, 500) * 4) / 4).astype(np.float32)  # heavy ties
    x = rng.uniform(0.0, 0.01, 400).astype(np.float32)
    x[17] = 1e4  # subtraction collapses the others into a few values
    yield x


def pin_score_rank_independent(orc):
    # rank by binary search in the sorted reported values (numpy FP32), against
    # the oracle's direct count; the record's lp and alternatives follow the
    # generation definitions already pinned above
    rng = np.random.default_rng(21)
    for x in _score_rows(rng):
        V = x.shape[0]
        targets = rng.integers(0, V, 12).astype(np.int32)
        targets[0] = int(np.argmax(x))
        r = orc.score(np.repeat(x[None, :], len(targets), 0), V, targets)
        lse = orc.lse(x)
        lps = (x - np.float32(lse)).astype(np.float32)
        desc = -np.sort(lps)[::-1]  # ascending copy of -lp for searchsorted
        ids, alt = orc.topk(x, 20, lse)
        for i, t in enumerate(targets):
            rec = r["records"][i]
            lpt = np.float32(x[t] - np.float32(lse))
            rank = int(np.searchsorted(desc, -lpt, side="left")) + 1
            assert rec[0] == t and rec[2] == rank, (int(t), int(rec[2]), rank)
            assert u32(rec[1]) == bits(np.float32(0.0) if lpt == 0 else lpt)
            assert list(rec[3::2][:len(ids)]) == list(ids)
            assert [u32(b) for b in rec[4::2][:len(ids)]] == [bits(v) for v in alt]
        assert r["records"][0][2] == 1  # the argmax has nothing strictly above it


def pin_score_collapse_closed_form(orc):
    # one logit of 3e7, the others in [0, 0.5]: lse rounds to 3e7 and every other
    # logprob rounds to -3e7 (half an ulp of 3e7 is 1), so each non-maximal
    # target has rank 2 and the alternatives after the maximum follow ascending id
    rng = np.random.default_rng(22)
    V = 200
    x = rng.uniform(0.0, 0.5, V).astype(np.float32)
    x[5] = np.float32(3e7)
    targets = np.array([5, 0, 199, 6], np.int32)
    r = orc.score(np.repeat(x[None, :], 4, 0), V, targets)["records"]
    assert r[0][2] == 1 and u32(r[0][1]) == bits(np.float32(0.0))
    for rec in r[1:]:
        assert rec[2] == 2 and u32(rec[1]) == bits(np.float32(-3e7))
        assert list(rec[3::2][:5]) == [5, 0, 1, 2, 3]


def pin_score_ties_and_invalid(orc):
    x = np.array([1.0, 4.0, 2.0, 4.0, 4.0, -0.0, 0.0], np.float32)
    V = 7
    targets = np.array([3, 4, 5, 6, -1, 7], np.int32)
    r = orc.score(np.repeat(x[None, :], 6, 0), V, targets)
    rec = r["records"]
    assert [int(v[2]) for v in rec[:4]] == [1, 1, 6, 6]  # equal values share a rank; -0 == +0
    assert list(rec[0][3::2][:7]) == [1, 3, 4, 2, 0, 5, 6] and list(rec[0][3::2][7:]) == [-1] * 13
    for bad in rec[4:]:
        assert bad[0] == -1 and bad[1] == NAN_BITS and bad[2] == 0
        assert all(int(v) == -1 for v in bad[3::2]) and all(int(v) == NAN_BITS for v in bad[4::2])
    assert r["status"] == 0x2  # the target 7 >= V; -1 is the ordinary invalid marker


# ----------------------------------------------------------------------------- commit clipping
#
# "mtp-design.md", a speculative round, step 4 and the paragraph after it: the
# emitted prefix of t tokens (1 <= t <= a+1) is clipped at an emitted EOS token
# (which stays emitted) and at the request's output budget; a request already at
# its limit takes no step.  The logprob writer reads only the emitted prefix.

CLIP_SENTINEL = 0x5EED5EED


def _clip_block():
    # four groups of k = 3 over a 40-lane vocabulary; every row has one planted
    # maximum (5.0), the rest in [0, 1)
    rng = np.random.default_rng(61)
    V = 40
    amax = [[7, 11, 13, 17], [7, 11, 13, 17], [21, 22, 23, 24], [30, 31, 32, 33]]
    x = rng.uniform(0.0, 1.0, (16, V)).astype(np.float32)
    for g in range(4):
        for j in range(4):
            x[4 * g + j, amax[g][j]] = 5.0
    drafts = np.full(16, -1, np.int32)
    drafts[0:3] = [7, 11, 13]       # group 0: every draft matches
    drafts[4:7] = [7, 12, 13]       # group 1: draft 1 misses (row 1's argmax is 11)
    drafts[8:11] = [21, 22, 23]     # group 2: every draft matches
    drafts[12:15] = [30, 31, 32]    # group 3: every draft matches
    return W.custom(x, V, [4, 4, 4, 4], drafts=drafts, top_k=[3, 3, 3, 3], k_max=3)


def pin_commit_clipping(orc):
    w = _clip_block()
    def run(eos, budget):
        rec = np.full((16, 258), CLIP_SENTINEL, np.int32)
        return orc.epilogue(w.logits_f32(), w.V, **w.inputs(), k_max=3, records=rec,
                            eos_tokens=None if eos is None else np.array(eos, np.int32),
                            budgets=None if budget is None else np.array(budget, np.int32))
    base = run(None, None)
    assert base["accepted"].tolist() == [3, 1, 3, 3] and base["rows_read"] == 4 + 2 + 4 + 4
    # budgets: at most that many tokens; 0 = at the limit (no step at all)
    r = run(None, [2, 1, 0, 9])
    assert r["accepted"].tolist() == [1, 0, -1, 3]
    assert r["emitted_tokens"].tolist() == [7, 11, -1, -1, 7, -1, -1, -1, -1, -1, -1, -1, 30, 31, 32, 33]
    assert r["rows_read"] == 2 + 1 + 0 + 4
    written = [not (row == CLIP_SENTINEL).all() for row in r["records"]]
    assert written == [True, True, False, False, True, False, False, False,
                       False, False, False, False, True, True, True, True]
    assert np.isnan(r["lse"][8:12]).all()
    # EOS: the emitted prefix ends at (and keeps) the first emitted EOS token,
    # whether it is an accepted draft, the correction or the bonus token
    r = run([11, 11, 24, 99], None)
    assert r["accepted"].tolist() == [1, 1, 3, 3]
    assert r["emitted_tokens"].tolist() == [7, 11, -1, -1, 7, 11, -1, -1, 21, 22, 23, 24, 30, 31, 32, 33]
    r = run([7, 12, 22, -1], [3, 9, 9, 2])
    # group 1: 12 is the rejected draft, never emitted; group 3: no EOS, budget 2
    assert r["accepted"].tolist() == [0, 1, 1, 1]
    assert r["emitted_tokens"].tolist() == [7, -1, -1, -1, 7, 11, -1, -1, 21, 22, -1, -1, 30, 31, -1, -1]
    assert r["rows_read"] == 1 + 2 + 2 + 2
    # k = 0 requests: a caller-sampled token is emitted as is (one token), not read
    x = np.zeros((2, 8), np.float32)
    w0 = W.custom(x, 8, [1, 1], sampled=[5, 5], requested=[0, 0], k_max=0)
    r0 = orc.epilogue(w0.logits_f32(), 8, **w0.inputs(), k_max=0, eos_tokens=np.array([5, 5], np.int32),
                      budgets=np.array([1, 0], np.int32))
    assert r0["accepted"].tolist() == [0, -1] and r0["emitted_tokens"].tolist() == [5, -1] and r0["rows_read"] == 0


# ----------------------------------------------------------------------------- stochastic chain verification
#
# "mtp-design.md", "Sampling correctness": accept a draft with probability
# min(1, p/q); on rejection draw the normalised positive residual max(p - q, 0);
# after full acceptance draw the bonus token from the target law.  The random
# numbers are inputs.


def _log_law(probs):
    return np.log(np.asarray(probs, np.float64)).astype(np.float32)


def pin_chain_closed_form(orc):
    # target rows with known laws at temperature 1, draft law q on row 0
    x = np.stack([_log_law([0.5, 0.3, 0.2]), _log_law([0.1, 0.1, 0.8])])
    q = np.array([[0.2, 0.6, 0.2], [0, 0, 0]], np.float32)
    def run(u0, r0, qq=q, d0=1):
        return orc.chain_verify(x, 3, [0, 2], [d0, -1], qq, [1.0], [u0, 0.0], [r0])
    r = run(0.4, 0.15)                      # 0.4 * 0.6 < 0.3: accepted; bonus from [.1, .1, .8]: 0.15 -> id 1
    assert r["accepted"].tolist() == [1] and r["emitted_tokens"].tolist() == [1, 1]
    r = run(0.4, 0.25)                      # bonus: 0.25 -> id 2
    assert r["emitted_tokens"].tolist() == [1, 2]
    r = run(0.6, 0.9)                       # 0.36 >= 0.3: rejected; residual [0.3, 0, 0] -> id 0
    assert r["accepted"].tolist() == [0] and r["emitted_tokens"].tolist() == [0, -1]
    q2 = np.array([[0.1, 0.8, 0.1], [0, 0, 0]], np.float32)  # residual [0.4, 0, 0.1], mass 0.5
    assert run(0.5, 0.7, q2)["emitted_tokens"].tolist() == [0, -1]    # 0.35 of 0.5 falls in lane 0
    assert run(0.5, 0.85, q2)["emitted_tokens"].tolist() == [2, -1]   # 0.425: past 0.4, lane 1 has none
    # temperature: logits (0, ln 3) at t = 0.5 give the law (0.1, 0.9)
    xt = np.array([[0.0, np.log(3.0)], [0.0, 0.0]], np.float32)
    qt = np.array([[0.5, 0.5], [0, 0]], np.float32)
    a = orc.chain_verify(xt, 2, [0, 2], [0, -1], qt, [0.5], [0.19, 0.0], [0.5])  # 0.19 * 0.5 < 0.1
    b = orc.chain_verify(xt, 2, [0, 2], [0, -1], qt, [0.5], [0.21, 0.0], [0.0])  # rejected: residual (0, 0.4)
    assert a["accepted"].tolist() == [1] and b["emitted_tokens"].tolist() == [1, -1]
    # two drafts: the first accepted, the second rejected
    x3 = np.stack([_log_law([0.5, 0.3, 0.2]), _log_law([0.2, 0.2, 0.6]), _log_law([1 / 3] * 3)])
    q3 = np.array([[0.2, 0.6, 0.2], [0.1, 0.1, 0.8], [0, 0, 0]], np.float32)
    r3 = orc.chain_verify(x3, 3, [0, 3], [1, 2, -1], q3, [1.0], [0.1, 0.9, 0.0], [0.25])
    assert r3["accepted"].tolist() == [1] and r3["emitted_tokens"].tolist() == [1, 0, -1]  # residual (.1, .1, 0)
    r3 = orc.chain_verify(x3, 3, [0, 3], [1, 2, -1], q3, [1.0], [0.1, 0.9, 0.0], [0.75])
    assert r3["emitted_tokens"].tolist() == [1, 1, -1]
    try:
        orc.chain_verify(xt, 2, [0, 2], [0, -1], qt, [0.0], [0.5, 0.0], [0.5])
    except RuntimeError:
        pass
    else:
        raise AssertionError("a temperature of 0 must be refused")


def pin_chain_preserves_target_law(orc):
    # The defining property: with d ~ q and u, r uniform, the first emitted
    # token follows p exactly, and the bonus token after an acceptance follows
    # the bonus row's law.  Every draft id is enumerated with weight q(d), u and
    # r run over midpoint grids of N points, so the frequencies must match the
    # laws to within about 1/N.
    V, N, t = 5, 160, 0.7
    rng = np.random.default_rng(81)
    x0 = rng.normal(0.0, 1.5, V).astype(np.float32)
    x1 = rng.normal(0.0, 1.5, V).astype(np.float32)
    q = rng.dirichlet(np.ones(V)).astype(np.float32)
    law = lambda x: np.exp(x / t - np.log(np.exp(x.astype(np.float64) / t).sum()))  # noqa: E731
    grid = (np.arange(N) + 0.5) / N
    d, ui, ri = np.meshgrid(np.arange(V), np.arange(N), np.arange(N), indexing="ij")
    d, ui, ri = d.ravel(), ui.ravel(), ri.ravel()
    G = d.size
    logits = np.empty((2 * G, V), np.float32)
    logits[0::2], logits[1::2] = x0, x1
    qq = np.zeros((2 * G, V), np.float32)
    qq[0::2] = q
    drafts = np.full(2 * G, -1, np.int32)
    drafts[0::2] = d
    u = np.zeros(2 * G, np.float32)
    u[0::2] = grid[ui]
    res = orc.chain_verify(logits, V, np.arange(G + 1) * 2, drafts, qq, np.full(G, t, np.float32), u,
                           grid[ri].astype(np.float32))
    wgt = q[d].astype(np.float64) / (N * N)
    first = res["emitted_tokens"][0::2]
    freq = np.bincount(first, weights=wgt, minlength=V)
    assert np.abs(freq - law(x0)).max() < 3.0 / N, (freq, law(x0))
    acc = res["accepted"] == 1
    bonus = np.bincount(res["emitted_tokens"][1::2][acc], weights=wgt[acc], minlength=V) / wgt[acc].sum()
    assert np.abs(bonus - law(x1)).max() < 3.0 / N, (bonus, law(x1))
    # the acceptance rate itself: sum over d of q(d) min(1, p(d)/q(d))
    rate = float(np.minimum(q.astype(np.float64), law(x0)).sum())
    assert abs(float(wgt[acc].sum()) - rate) < 2.0 / N


ALL_PINS = [pin_golden_rows, pin_golden_groups, pin_brute_force, pin_lse_independent,
            pin_two_value_closed_form, pin_sum_exp_invariant, pin_pad_exclusion, pin_id_passthrough,
            pin_acceptance_prefixes, pin_tiny_workload, pin_status_bits, pin_score_rank_independent,
            pin_score_collapse_closed_form, pin_score_ties_and_invalid, pin_commit_clipping,
            pin_chain_closed_form, pin_chain_preserves_target_law]
