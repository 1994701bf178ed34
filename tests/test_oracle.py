"""CPU tests of the oracle against its pins, plus revert-checks.

A revert-check plants one plausible mistake in a copy of the oracle source
(on the CPU), builds it, and requires that at least one pin fails.
"""
import os
import shutil

import numpy as np
import pytest

import oracle
import oracle_pins as P


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_pin_wide_tie(orc):
    P.pin_wide_tie(orc)


def test_threads_match_single(orc):
    import workloads as W
    w = W.spec(groups=6, V=20_000, Vp=20_008)
    a = orc.epilogue(w.logits_f32(), w.V, **w.inputs(), k_max=w.k_max, threads=1)
    b = orc.epilogue(w.logits_f32(), w.V, **w.inputs(), k_max=w.k_max, threads=4)
    for key in ("records", "accepted", "emitted_tokens", "status", "rows_read"):
        assert np.array_equal(np.asarray(a[key]), np.asarray(b[key])), key


MUTANTS = {
    "tie_break_reversed": ("return a.lp > b.lp; });",
                           "return a.lp > b.lp || (a.lp == b.lp && a.id > b.id); });"),
    "no_signed_zero_normalisation": ("if (r == 0.0f) r = 0.0f;", ""),
    "argmax_last_of_ties": ("if (x[v] > x[best]) best", "if (x[v] >= x[best]) best"),
    "lse_float_sum": ("double s = 0.0;\n    for (int64_t v = 0; v < V; ++v) s += std::exp((double)x[v] - m);",
                      "float s = 0.0f;\n    for (int64_t v = 0; v < V; ++v) s += (float)std::exp((double)x[v] - m);"),
    "lse_drop_max": ("double lse = m + std::log(s);", "double lse = std::log(s);"),
    "logprob_sign": ("volatile float d = x - lse;", "volatile float d = lse - x;"),
    "accepted_off_by_one": ("io.accepted[g] = j;", "io.accepted[g] = j + 1;"),
    "pads_included": ("const int32_t amax = orc_argmax(x, io.V);", "const int32_t amax = orc_argmax(x, io.Vp);"),
    "pads_in_lse": ("const float lse = orc_lse(x, io.V);", "const float lse = orc_lse(x, io.Vp);"),
    "unused_pair_id_zero": ("rec[2 + 2 * i] = -1;", "rec[2 + 2 * i] = 0;"),
    "rejected_rows_not_cleared": ("for (int32_t jj = j + 1; jj <= k; ++jj) io.emitted_tokens[(int64_t)r0 + jj] = -1;", ""),
    "reads_past_prefix": ("            break;\n        }\n    }\n    sh.rows_read", "        }\n    }\n    sh.rows_read"),
    "topk_by_raw_logit": ("all[(size_t)v] = Pair{orc_logprob(x[v], lse), (int32_t)v};",
                          "all[(size_t)v] = Pair{x[v], (int32_t)v};"),
    "unflagged_k0_read": ("const bool must_read = flagged || k >= 1 || sampled < 0;",
                          "const bool must_read = true;"),
    "rank_counts_ties": ("if (orc_logprob(x[v], lse) > lp) ++greater;", "if (orc_logprob(x[v], lse) >= lp) ++greater;"),
    "rank_before_rounding": ("if (orc_logprob(x[v], lse) > lp) ++greater;",
                             "if ((double)x[v] - (double)lse > (double)lp) ++greater;"),
    "rank_zero_based": ("    return 1 + greater;", "    return greater;"),
    "invalid_rank_one": ("        rec[2] = 0;", "        rec[2] = 1;"),
    "invalid_alt_id_zero": ("            rec[3 + 2 * i] = -1;", "            rec[3 + 2 * i] = 0;"),
    "budget_off_by_one": ("|| j + 1 >= budget;", "|| j >= budget;"),
    "eos_ignored": ("const bool clipped = (eos >= 0 && chosen == eos) || j + 1 >= budget;",
                    "const bool clipped = j + 1 >= budget;"),
    "at_limit_still_steps": ("    if (budget <= 0) {", "    if (budget < 0) {"),
    "chain_accept_ratio_inverted": ("if ((double)u[row] * qd < pd) {", "if ((double)u[row] * pd < qd) {"),
    "chain_residual_abs": ("w[(size_t)v] = std::max(p[(size_t)v] - (double)q[v], 0.0);",
                           "w[(size_t)v] = std::fabs(p[(size_t)v] - (double)q[v]);"),
    "chain_reject_draws_target": ("last = draw(mass > 0.0 ? w : p, (double)r[g]);", "last = draw(p, (double)r[g]);"),
    "chain_temperature_ignored": ("target_law(logits + row * Vp, V, t, p);", "target_law(logits + row * Vp, V, 1.0, p);"),
    "eos_not_emitted": ("        io.emitted_tokens[row] = chosen;\n",
                        "        io.emitted_tokens[row] = (eos >= 0 && chosen == eos) ? -1 : chosen;\n"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_revert_check(name, tmp_path):
    find, repl = MUTANTS[name]
    here = os.path.dirname(oracle.__file__)
    src = open(os.path.join(here, "lp_oracle.cpp")).read()
    assert src.count(find) == 1, f"mutation anchor not found once: {name}"
    mdir = tmp_path / name
    mdir.mkdir()
    shutil.copy(os.path.join(here, "lp_oracle.h"), mdir / "lp_oracle.h")
    (mdir / "lp_oracle.cpp").write_text(src.replace(find, repl))
    lib = oracle.build(force=True, src=str(mdir / "lp_oracle.cpp"), out=str(mdir / "libmut.so"))
    mut = oracle.load(lib)
    caught = []
    for pin in P.ALL_PINS + [P.pin_wide_tie]:
        try:
            pin(mut)
        except Exception as e:  # noqa: BLE001 - any failure counts as caught
            caught.append((pin.__name__, type(e).__name__))
            break
    assert caught, f"mutant {name} passed every pin"
