"""Helpers: run a workload through the C-ABI (CUDA path) and through the oracle,
and compare the two by the parity rule of the epilogue:

  * bit-exact: accepted counts, emitted tokens, chosen ids, explicit ids and
    their order, the number of natural alternatives, unused pairs (-1, NaN
    bits), untouched records of rows that are not written, status bits;
  * |delta| <= 2e-5 on every FP32 logprob and on lse, widened to one FP32 ulp
    of the row's lse where that spacing is coarser (|lse| >= 256): there two
    correctly rounded FP32 results of nearly the same real differ by an ulp;
  * natural-alternative ids bit-exact, except where the reported values of the
    candidates differ by less than the tolerance: there, any order consistent
    with (logprob descending, id ascending) on the CUDA path's own values is
    accepted, including which id fills the K-th slot;
  * where the CUDA path's lse equals the oracle's bit for bit, the whole record
    must be bit-identical.
"""
from __future__ import annotations

import numpy as np

import oracle
import workloads as W

TOL = 2e-5
NAN_BITS = 0x7FC00000
SENTINEL = 0x5EED5EED
LSE_SENTINEL = -12345.0


def to_device(w: W.Workload):
    import torch
    if w.dtype == "bf16":
        logits = torch.from_numpy(w.logits.view(np.int16)).view(torch.bfloat16)
    else:
        logits = torch.from_numpy(w.logits)
    dev = torch.device("cuda", 0)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)  # noqa: E731
    G = w.groups
    return dict(
        logits=logits.to(dev).contiguous(),
        group_indptr=t(w.group_indptr),
        draft_tokens=t(w.draft_tokens),
        sampled_tokens=t(w.sampled_tokens if G else np.zeros(1)),
        requested=t(w.requested if G else np.zeros(1)),
        top_k=t(w.top_k if G else np.zeros(1)),
        token_ids=t(w.token_ids.reshape(-1) if G else np.zeros(128)),
        id_counts=t(w.id_counts if G else np.zeros(1)),
    )


def make_plan(w: W.Workload, **kw):
    import logprob_epilogue_gb300 as lpe
    args = dict(max_rows=max(w.rows, 1), max_groups=max(w.groups, 1), k_max=w.k_max, V=w.V, V_padded=w.Vp,
                dtype=w.dtype, k_alt_max=20, max_ids=128, device=0)
    args.update(kw)
    return lpe.Plan(**args)


def run_gpu(w: W.Workload, plan=None, dev_inputs=None, poison=False, runs=1, eos_tokens=None, budgets=None):
    """Runs the CUDA path; returns numpy outputs and the plan.  ``eos_tokens`` /
    ``budgets`` ([groups] int32, optional) attach commit clipping."""
    import torch
    if plan is None:
        plan = make_plan(w)
    dev = torch.device("cuda", 0)
    d = dev_inputs if dev_inputs is not None else to_device(w)
    rows, G = w.rows, w.groups
    out = dict(
        records=torch.full((max(rows, 1), 258), SENTINEL, dtype=torch.int32, device=dev),
        accepted=torch.full((max(G, 1),), -7, dtype=torch.int32, device=dev),
        emitted_tokens=torch.full((max(rows, 1),), -7, dtype=torch.int32, device=dev),
        lse_out=torch.full((max(rows, 1),), LSE_SENTINEL, dtype=torch.float32, device=dev),
        status=torch.full((1,), -1, dtype=torch.int32, device=dev),
    )
    plan.bind(**d, **out)
    if eos_tokens is not None or budgets is not None:
        ti = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)  # noqa: E731
        clip = (ti(eos_tokens), ti(budgets))
        plan.bind_clip(eos_tokens=clip[0], budgets=clip[1])
    for _ in range(runs):
        if poison:
            plan.poison_scratch()
        plan.run()
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy() for k, v in out.items()}
    res["records"] = res["records"][:rows]
    res["accepted"] = res["accepted"][:G]
    res["emitted_tokens"] = res["emitted_tokens"][:rows]
    res["lse"] = res["lse_out"][:rows]
    res["status"] = int(res["status"].view(np.uint32)[0])
    res["tiles_read"] = plan.tiles_read(rows)
    return res, plan


def run_oracle(w: W.Workload, threads: int = 8, eos_tokens=None, budgets=None):
    sentinel = np.full((w.rows, 258), SENTINEL, np.int32)
    return oracle.epilogue(w.logits_f32(), w.V, **w.inputs(), k_max=w.k_max, records=sentinel, threads=threads,
                           eos_tokens=eos_tokens, budgets=budgets)


def _f(bits) -> np.float32:
    return np.array([bits], np.int32).view(np.float32)[0]


def compare(w: W.Workload, gpu: dict, orc: dict, check_invariant: bool = True) -> dict:
    """Asserts parity; returns a few statistics."""
    stats = {"rows_written": 0, "near_tie_swaps": 0, "strict_rows": 0, "max_lp_err": 0.0, "max_lse_err": 0.0}
    assert gpu["status"] == orc["status"], (hex(gpu["status"]), hex(orc["status"]))
    assert np.array_equal(gpu["accepted"], orc["accepted"]), "accepted"
    assert np.array_equal(gpu["emitted_tokens"], orc["emitted_tokens"]), "emitted_tokens"
    rows_x = None
    for r in range(w.rows):
        orec = orc["records"][r]
        grec = gpu["records"][r]
        written = not (orec == SENTINEL).all()
        if not written:
            assert (grec == SENTINEL).all(), f"row {r}: record written but the oracle wrote none"
            assert gpu["lse"][r] == np.float32(LSE_SENTINEL), f"row {r}: lse written"
            continue
        stats["rows_written"] += 1
        olse, glse = np.float32(orc["lse"][r]), np.float32(gpu["lse"][r])
        tol = row_tol(olse)
        lse_err = abs(float(olse) - float(glse))
        stats["max_lse_err"] = max(stats["max_lse_err"], lse_err)
        assert lse_err <= tol, f"row {r}: lse {glse} vs {olse}"
        strict = olse.view(np.uint32) == glse.view(np.uint32)
        if strict:
            stats["strict_rows"] += 1
            assert np.array_equal(grec, orec), f"row {r}: lse identical but records differ at " \
                f"{np.flatnonzero(grec != orec)[:8]}"
            continue
        # chosen pair
        assert grec[0] == orec[0], f"row {r}: chosen id"
        _cmp_lp(r, "chosen", grec[1], orec[1], stats, tol)
        g = int(np.flatnonzero(np.asarray(w.group_indptr) <= r)[-1]) if w.groups else 0
        explicit = int(w.requested[g]) != 0 and int(w.id_counts[g]) != 0
        gids, oids = grec[2::2], orec[2::2]
        glp, olp = grec[3::2], orec[3::2]
        n_o = int((oids != -1).sum()) if not explicit else int(min(max(int(w.id_counts[g]), 0), 128))
        if explicit:
            assert np.array_equal(gids, oids), f"row {r}: explicit ids"
            for i in range(n_o):
                _cmp_lp(r, f"id[{i}]", glp[i], olp[i], stats, tol)
        else:
            n_g = int((gids != -1).sum())
            assert n_g == n_o, f"row {r}: {n_g} natural alternatives vs {n_o}"
            if rows_x is None or rows_x[0] != r:
                rows_x = (r, w.logits_f32(r))
            x = rows_x[1]
            gv = [_f(b) for b in glp[:n_g]]
            for i in range(n_g):
                _cmp_lp(r, f"alt[{i}]", glp[i], olp[i], stats, tol)
                if gids[i] != oids[i]:
                    # allowed only as a near-tie: the oracle's own value at the CUDA id
                    ov = oracle.logprob(x[gids[i]], olse)
                    assert abs(float(ov) - float(_f(olp[i]))) <= tol, \
                        f"row {r}: alt[{i}] id {gids[i]} vs {oids[i]} not a near tie"
                    stats["near_tie_swaps"] += 1
            # self-consistency of the CUDA list: (lp desc, id asc), distinct ids in range
            assert len(set(gids[:n_g].tolist())) == n_g and ((gids[:n_g] >= 0) & (gids[:n_g] < w.V)).all()
            for i in range(n_g - 1):
                assert gv[i] > gv[i + 1] or (gv[i] == gv[i + 1] and gids[i] < gids[i + 1]), \
                    f"row {r}: CUDA alternatives out of order at {i}"
        # unused pairs
        assert (gids[n_o:] == -1).all() and (glp[n_o:] == NAN_BITS).all(), f"row {r}: unused pairs"
        if check_invariant:
            xr = w.logits_f32(r)[:w.V].astype(np.float64)
            total = float(np.exp(xr - np.float64(glse)).sum())
            assert abs(total - 1.0) <= 1e-5, f"row {r}: sum exp(lp) = {total}"
    return stats


def row_tol(lse) -> float:
    """2e-5, or one FP32 ulp of lse where the format is coarser than that: two
    correctly rounded lse values of nearly the same real differ by one ulp, and
    then fl32(x - lse) differs by at most that ulp (both roundings of the
    subtraction land on the same grid when |x - lse| is in lse's binade, and
    are exact or finer below it)."""
    return max(TOL, float(np.spacing(np.abs(np.float32(lse)))))


def _cmp_lp(r, what, gb, ob, stats, tol=TOL):
    gb, ob = int(gb), int(ob)
    if (ob & 0xFFFFFFFF) == NAN_BITS:
        assert (gb & 0xFFFFFFFF) == NAN_BITS, f"row {r}: {what} expected NaN bits"
        return
    g, o = _f(gb), _f(ob)
    err = abs(float(g) - float(o))
    stats["max_lp_err"] = max(stats["max_lp_err"], err)
    assert err <= tol, f"row {r}: {what} lp {g} vs {o}"
    if float(o) == 0.0:
        assert (gb & 0xFFFFFFFF) != 0x80000000, f"row {r}: {what} -0 not normalised"


def lpe_tile_elems(dtype: str) -> int:
    """Vocabulary tile of the CUDA path: 32 KiB of logits."""
    return 32768 // (2 if dtype == "bf16" else 4)


def expected_tiles(w: W.Workload, orc: dict) -> np.ndarray:
    """Tiles each row must read: all tiles of rows the path reads, 0 elsewhere
    (the exact count of a plan that reads no row past a prefix)."""
    te = lpe_tile_elems(w.dtype)
    T = (w.V + te - 1) // te
    tiles = np.zeros(w.rows, np.int32)
    for g in range(w.groups):
        r0, r1 = int(w.group_indptr[g]), int(w.group_indptr[g + 1])
        k = r1 - r0 - 1
        need = int(w.requested[g]) != 0 or k >= 1 or int(w.sampled_tokens[g]) < 0
        if not need:
            continue
        a = int(orc["accepted"][g])
        tiles[r0:r0 + a + 1] = T
    return tiles


def check_tiles(w: W.Workload, orc: dict, tiles: np.ndarray, strict: bool) -> None:
    """Tiles read per row.  Strict plans read exactly the prefix rows.  With
    read-ahead, the prefix rows are read in full, the first row past a verify
    group's prefix may be read in part or in full (it was the successor of a
    row being decided), and no other row is read."""
    want = expected_tiles(w, orc)
    if strict:
        assert np.array_equal(tiles, want), "tiles read per row"
        return
    T = int(want.max()) if want.size and want.max() > 0 else 0
    allowed = want.copy()
    for g in range(w.groups):
        r0, r1 = int(w.group_indptr[g]), int(w.group_indptr[g + 1])
        if want[r0] == 0:
            continue
        nxt = r0 + int(orc["accepted"][g]) + 1
        if nxt < r1:
            allowed[nxt] = T
    prefix = want > 0
    assert np.array_equal(tiles[prefix], want[prefix]), "prefix rows read in full"
    assert ((tiles >= 0) & (tiles <= allowed)).all(), "no row read beyond the one after a prefix"



# ----------------------------------------------------------------- prompt scoring

SCORE_WORDS = 43


def run_gpu_score(w: W.Workload, targets, plan=None, poison=False, runs=1):
    """Prompt scoring on the CUDA path: numpy records [rows, 43], lse, status."""
    import torch
    if plan is None:
        plan = make_plan(w)
    dev = torch.device("cuda", 0)
    d = to_device(w)
    rows = w.rows
    tg = torch.from_numpy(np.ascontiguousarray(targets, np.int32)).to(dev)
    rec = torch.full((max(rows, 1), SCORE_WORDS), SENTINEL, dtype=torch.int32, device=dev)
    lse = torch.full((max(rows, 1),), LSE_SENTINEL, dtype=torch.float32, device=dev)
    st = torch.full((1,), -1, dtype=torch.int32, device=dev)
    for _ in range(runs):
        if poison:
            plan.poison_scratch()
        plan.score(logits=d["logits"], target_tokens=tg, records=rec, status=st, lse_out=lse)
    torch.cuda.synchronize()
    res = dict(records=rec.cpu().numpy()[:rows], lse=lse.cpu().numpy()[:rows],
               status=int(st.cpu().numpy().view(np.uint32)[0]), tiles_read=plan.tiles_read(rows))
    return res, plan


def run_oracle_score(w: W.Workload, targets, threads: int = 8):
    return oracle.score(w.logits_f32(), w.V, np.asarray(targets, np.int32), threads=threads)


def compare_score(w: W.Workload, targets, gpu: dict, orc: dict) -> dict:
    """Parity of prompt-scoring records.  The integer words are bit-exact; the
    ones FP32 decides (the target's lp bits, its rank, the alternatives and
    their order) are decided on both sides with the CUDA path's lse, which must
    itself be within the tolerance of the oracle's."""
    stats = {"scored": 0, "strict_rows": 0, "max_lse_err": 0.0, "max_lp_err": 0.0, "ranks_above_1": 0}
    assert gpu["status"] == orc["status"], (hex(gpu["status"]), hex(orc["status"]))
    for r in range(w.rows):
        t = int(targets[r])
        grec, orec = gpu["records"][r], orc["records"][r]
        if not (0 <= t < w.V):
            assert np.array_equal(grec, orec), f"row {r}: invalid-target record"
            assert gpu["lse"][r] == np.float32(LSE_SENTINEL), f"row {r}: lse written for an unread row"
            continue
        stats["scored"] += 1
        olse, glse = np.float32(orc["lse"][r]), np.float32(gpu["lse"][r])
        tol = row_tol(olse)
        err = abs(float(olse) - float(glse))
        stats["max_lse_err"] = max(stats["max_lse_err"], err)
        assert err <= tol, f"row {r}: lse {glse} vs {olse}"
        if olse.view(np.uint32) == glse.view(np.uint32):
            stats["strict_rows"] += 1
            assert np.array_equal(grec, orec), f"row {r}: lse identical but records differ at " \
                f"{np.flatnonzero(grec != orec)[:8]}"
            continue
        x = w.logits_f32(r)[:w.V]
        assert grec[0] == t, f"row {r}: target id"
        lp = oracle.logprob(x[t], glse)
        assert (int(grec[1]) & 0xFFFFFFFF) == int(np.float32(lp).view(np.uint32)), f"row {r}: lp bits"
        _cmp_lp(r, "target", grec[1], orec[1], stats, tol)
        assert grec[2] == oracle.rank(x, glse, lp), f"row {r}: rank {grec[2]} vs {oracle.rank(x, glse, lp)}"
        ids, lps = oracle.topk(x, 20, glse)
        n = ids.size
        assert np.array_equal(grec[3::2][:n], ids), f"row {r}: alternative ids"
        assert np.array_equal(grec[4::2][:n].view(np.uint32), lps.view(np.uint32)), f"row {r}: alternative lps"
        assert (grec[3::2][n:] == -1).all() and (grec[4::2][n:] == NAN_BITS).all(), f"row {r}: unused pairs"
        for i in range(n):
            _cmp_lp(r, f"alt[{i}]", grec[4 + 2 * i], orec[4 + 2 * i], stats, tol)
    for r in range(w.rows):
        if 0 <= int(targets[r]) < w.V and gpu["records"][r][2] > 1:
            stats["ranks_above_1"] += 1
    return stats
