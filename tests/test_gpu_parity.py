"""CUDA path vs the CPU oracle, element by element, through the C ABI."""
import os

import numpy as np
import pytest

import parity as PT
import workloads as W

pytestmark = pytest.mark.gpu
THREADS = os.cpu_count() or 8


def _check(w, read_ahead=False, **kw):
    if read_ahead and "plan" not in kw:
        kw["plan"] = PT.make_plan(w, read_ahead=True)
    gpu, plan = PT.run_gpu(w, **kw)
    orc = PT.run_oracle(w, THREADS)
    stats = PT.compare(w, gpu, orc)
    PT.check_tiles(w, orc, gpu["tiles_read"], strict=not read_ahead)
    plan.close()
    return gpu, orc, stats


# ----------------------------------------------------------------- workloads

SMALL = {
    "tiny": lambda: W.tiny(),
    "decode": lambda: W.decode(rows=16),
    "spec": lambda: W.spec(groups=12),
    "large": lambda: W.large(groups=12),
    "wide": lambda: W.wide(),
}


@pytest.mark.parametrize("read_ahead", [False, True], ids=["prefix_only", "read_ahead"])
@pytest.mark.parametrize("name", list(SMALL))
def test_workload_small(name, read_ahead):
    _, orc, stats = _check(SMALL[name](), read_ahead=read_ahead)
    assert stats["rows_written"] > 0


@pytest.mark.parametrize("name", ["decode", "spec", "large"])
def test_workload_full_size(name):
    w = W.make(name)
    gpu, orc, stats = _check(w)
    # the benchmark's launch configuration is the plan's default one
    assert stats["rows_written"] > 0


def test_tiny_hand_checked():
    w = W.tiny()
    gpu, plan = PT.run_gpu(w)
    plan.close()
    assert gpu["accepted"].tolist() == [2, 0, 0]
    assert gpu["emitted_tokens"][:3].tolist() == [int(w.draft_tokens[0]), int(w.draft_tokens[1]),
                                                  int(w.planted_argmax[2])]
    assert gpu["tiles_read"].tolist() == [1, 1, 1, 0, 1, 0]
    # with read-ahead only row 3, the successor of the rejecting row 2, may also be read
    gpu2, plan = PT.run_gpu(w, plan=PT.make_plan(w, read_ahead=True))
    plan.close()
    for key in ("records", "accepted", "emitted_tokens", "lse"):
        assert np.array_equal(gpu[key], gpu2[key]), key
    t = gpu2["tiles_read"].tolist()
    assert t[:3] == [1, 1, 1] and t[3] in (0, 1) and t[4:] == [1, 0]


def test_wide_tie_all_accepted():
    w = W.wide()
    gpu, _ = PT.run_gpu(w)
    assert gpu["accepted"].tolist() == [3]
    x = w.logits_f32(3)
    tied = np.sort(np.flatnonzero(x[:w.V] == np.float32(16.0)))
    assert gpu["records"][3][2:42:2].tolist() == tied[:20].tolist()


# ----------------------------------------------------------------- adversarial rows

def _one_group(rows, V, *, dtype="f32", Vp=None, k=None, drafts=None, top_k=20, ids=None, requested=1,
               sampled=-1):
    rows = np.asarray(rows, np.float32)
    n = rows.shape[0]
    k = n - 1 if k is None else k
    return W.custom(rows, V, [n], dtype=dtype, Vp=Vp, drafts=drafts, top_k=[top_k],
                    token_ids=[ids] if ids is not None else None,
                    id_counts=[len(ids)] if ids is not None else None, requested=[requested],
                    sampled=[sampled], k_max=max(k, 0))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_subtraction_ties_across_tiles(dtype):
    rng = np.random.default_rng(3)
    V = 30_000
    x = rng.uniform(0.0, 0.01, V).astype(np.float32)
    x[rng.integers(0, V)] = 1e4
    w = _one_group(x[None, :], V, dtype=dtype, Vp=V + (8 if dtype == "bf16" else 0))
    _check(w)


def test_subtraction_ties_hidden_below_tile_top32():
    # one tile holds many logits that collapse to the same logprob, with small ids
    rng = np.random.default_rng(4)
    V = 40_000
    x = rng.normal(-30.0, 1.0, V).astype(np.float32)
    x[0] = 2000.0
    x[1:5000] = (rng.uniform(0, 0.003, 4999) + 1990.0).astype(np.float32)
    _check(_one_group(x[None, :], V))


def test_exact_tie_split_across_tiles():
    rng = np.random.default_rng(5)
    V = 100_000
    x = rng.normal(0, 1, V).astype(np.float32)
    ids = rng.choice(V, 64, replace=False)
    x[ids] = 16.0
    _check(_one_group(x[None, :], V, dtype="bf16"))


def test_tie_straddles_cutoff():
    rng = np.random.default_rng(6)
    V = 50_000
    x = rng.normal(0, 1, V).astype(np.float32)
    top = rng.choice(V, 40, replace=False)
    x[top[:10]] = np.arange(20, 30, dtype=np.float32)
    x[top[10:]] = 7.0
    _check(_one_group(x[None, :], V))


@pytest.mark.parametrize("off_grid", [False, True], ids=["bf16_grid", "one_off_grid"])
def test_fp32_ties_on_the_bf16_grid(off_grid):
    # FP32 logits that are all BF16-representable (as when computed in BF16)
    # select each tile's best 32 on 32-bit keys; one value off the grid sends
    # its tile back to 64-bit keys.  Heavy ties at the top, across 4 tiles.
    rng = np.random.default_rng(7)
    V = 30_000
    x = np.round(rng.normal(0, 1, V) * 2.0) / 2.0  # steps of 0.5: exact in BF16
    top = rng.choice(V, 80, replace=False)
    x[top] = 6.0
    x[top[:5]] = 6.5
    if off_grid:
        x[top[5]] = 6.0 + 2.0 ** -10  # between BF16 neighbours
    x = x.astype(np.float32)
    w = _one_group(np.stack([x, x[::-1].copy()]), V, drafts=[int(np.argmax(x)), -1])
    _check(w)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_constant_row(dtype):
    V = 30_000
    x = np.zeros((1, V), np.float32)
    _check(_one_group(x, V, dtype=dtype, Vp=V + (8 if dtype == "bf16" else 0)))


def test_signed_zero_maximum():
    V = 9000
    x = np.full(V, -3.0, np.float32)
    x[8500] = -0.0
    x[8200] = 0.0
    x[100] = -0.0
    w = _one_group(np.stack([x, x]), V, drafts=[100, -1])
    gpu, _, _ = _check(w)
    assert gpu["emitted_tokens"].tolist() == [100, 100]


@pytest.mark.parametrize("V,Vp,dtype", [(10_001, 10_008, "bf16"), (10_001, 10_004, "f32"), (7, 8, "bf16"),
                                        (1, 4, "f32"), (33, 40, "bf16"), (8192, 8192, "f32"),
                                        (8193, 8200, "bf16"), (16_385, 16_388, "f32")])
def test_ragged_vocabularies(V, Vp, dtype):
    rng = np.random.default_rng(V)
    rows = rng.normal(0, 2, (3, V)).astype(np.float32)
    rows[:, rng.integers(0, V)] = 20.0
    w = W.custom(rows, V, [2, 1], dtype=dtype, Vp=Vp, drafts=[int(np.argmax(rows[0])), -1, -1],
                 top_k=[20, 5], k_max=1)
    _check(w)


@pytest.mark.parametrize("a", [0, 1, 7, 15])
@pytest.mark.parametrize("read_ahead", [False, True], ids=["prefix_only", "read_ahead"])
def test_acceptance_prefixes_k15(a, read_ahead):
    rng = np.random.default_rng(100 + a)
    k, V = 15, 20_000
    rows = rng.normal(0, 1, (k + 1, V)).astype(np.float32)
    am = rng.integers(0, V, k + 1)
    rows[np.arange(k + 1), am] = 8.0
    drafts = np.full(k + 1, -1, np.int32)
    drafts[:k] = am[:k]
    if a < k:
        drafts[a] = (am[a] + 1) % V
    w = _one_group(rows, V, drafts=drafts, top_k=3)
    gpu, _, _ = _check(w, read_ahead=read_ahead)
    assert int(gpu["accepted"][0]) == a


def test_explicit_ids_edges_and_errors():
    rng = np.random.default_rng(8)
    V = 12_345
    rows = rng.normal(0, 2, (2, V)).astype(np.float32)
    ids = [0, V - 1, 5, -1, V, 77]
    w = W.custom(rows, V, [1, 1], dtype="bf16", Vp=12_352, top_k=[0, 25],
                 token_ids=[ids, None], id_counts=[len(ids), 0], k_max=0)
    gpu, orc, _ = _check(w)
    assert gpu["status"] == (0x1 | 0x4)


def test_flags_and_unread_groups():
    rng = np.random.default_rng(9)
    V = 5000
    rows = rng.normal(0, 1, (6, V)).astype(np.float32)
    # g0 unflagged k=0 with a token (never read), g1 unflagged k=0 argmax (read, no record),
    # g2 flagged K=0 (lse only), g3 unflagged verify group k=2, g4 flagged with a bad token
    w = W.custom(rows, V, [1, 1, 1, 2, 1], sampled=[17, -1, 3, -1, V + 5], requested=[0, 0, 1, 0, 1],
                 top_k=[20, 20, 0, 20, 20], drafts=[-1, -1, -1, int(np.argmax(rows[3])), -1, -1], k_max=1)
    gpu, orc, _ = _check(w)
    assert gpu["tiles_read"][0] == 0
    assert gpu["status"] == 0x2


def test_poisoned_scratch_and_repeated_runs():
    w = W.spec(groups=6)
    gpu1, plan = PT.run_gpu(w, plan=PT.make_plan(w, read_ahead=True))
    gpu2, _ = PT.run_gpu(w, plan=plan, poison=True, runs=3)
    for key in ("records", "accepted", "emitted_tokens", "lse"):
        assert np.array_equal(gpu1[key], gpu2[key]), key
    # read-ahead may differ from run to run; the prefix rows may not
    orc = PT.run_oracle(w, THREADS)
    PT.check_tiles(w, orc, gpu1["tiles_read"], False)
    PT.check_tiles(w, orc, gpu2["tiles_read"], False)
    plan.close()


@pytest.mark.parametrize("name", ["large", "spec"])
def test_decisions_stable_over_back_to_back_runs(name):
    # Each acceptance decision reads the row's best key, which the compute warps
    # of other CTAs update; a decision taken before the last update has landed
    # picks a wrong argmax.  1,000 back-to-back runs on the full-size block (no
    # L2 flush, scratch poisoned before every third) must each give the
    # oracle's accepted counts and emitted tokens.
    import torch
    w = W.make(name)
    orc = PT.run_oracle(w, THREADS)
    d = PT.to_device(w)
    dev = torch.device("cuda", 0)
    rows, G, reps = w.rows, w.groups, 1000
    out = dict(records=torch.zeros((rows, 258), dtype=torch.int32, device=dev),
               accepted=torch.zeros(G, dtype=torch.int32, device=dev),
               emitted_tokens=torch.zeros(rows, dtype=torch.int32, device=dev),
               lse_out=torch.zeros(rows, dtype=torch.float32, device=dev),
               status=torch.zeros(1, dtype=torch.int32, device=dev))
    plan = PT.make_plan(w)
    plan.bind(**d, **out)
    accs = torch.zeros((reps, G), dtype=torch.int32, device=dev)
    ems = torch.zeros((reps, rows), dtype=torch.int32, device=dev)
    sts = torch.zeros(reps, dtype=torch.int32, device=dev)
    for r in range(reps):
        if r % 3 == 0:
            plan.poison_scratch()
        plan.run()
        accs[r].copy_(out["accepted"])
        ems[r].copy_(out["emitted_tokens"])
        sts[r].copy_(out["status"][0])
    torch.cuda.synchronize()
    A, E, S = accs.cpu().numpy(), ems.cpu().numpy(), sts.cpu().numpy()
    plan.close()
    assert (S == 0).all()
    bad = np.flatnonzero((A != orc["accepted"][None, :]).any(1) | (E != orc["emitted_tokens"][None, :]).any(1))
    assert bad.size == 0, f"{bad.size} of {reps} runs differ from the oracle (first: run {bad[:5].tolist()})"


@pytest.mark.parametrize("name", ["spec", "large"])
def test_run_beside_a_kernel_holding_half_the_gpu(name):
    # Another kernel, on another stream, holds half the multiprocessors for
    # 150 ms, longer than the plan's 30 ms limit on every device wait, so the
    # stream kernel starts with only part of its grid resident.  The resident
    # CTAs must do all the work: same outputs as the oracle, status 0.
    import torch
    import logprob_epilogue_gb300 as lpe
    w = {"spec": lambda: W.spec(groups=24), "large": lambda: W.large(groups=16)}[name]()
    dev = torch.device("cuda", 0)
    d = PT.to_device(w)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    side = torch.cuda.Stream(dev)
    lpe.debug_occupy(0, sms // 2, 150_000_000, side)
    gpu, plan = PT.run_gpu(w, plan=PT.make_plan(w, timeout_ns=30_000_000), dev_inputs=d)
    side.synchronize()
    orc = PT.run_oracle(w, THREADS)
    assert gpu["status"] == 0
    PT.compare(w, gpu, orc)
    PT.check_tiles(w, orc, gpu["tiles_read"], strict=True)
    plan.close()


def test_malformed_groups_write_nothing():
    x = np.zeros((3, 100), np.float32)
    w = W.custom(x, 100, [2, 1], k_max=0)   # a group of 2 rows with k_max 0
    gpu, _ = PT.run_gpu(w)
    assert gpu["status"] == 0x8
    assert (gpu["emitted_tokens"] == -7).all() and (gpu["records"] == PT.SENTINEL).all()
    assert (gpu["tiles_read"] == 0).all()


def test_no_groups():
    x = np.zeros((2, 64), np.float32)
    w = W.custom(x, 64, [], k_max=0)
    gpu, _ = PT.run_gpu(w)
    assert gpu["status"] == 0 and (gpu["tiles_read"] == 0).all()


def test_forced_timeout_is_reported_and_context_survives():
    w = W.spec(groups=2, V=20_000, Vp=20_000)
    plan = PT.make_plan(w, debug_force_timeout=True, timeout_ns=2_000_000)
    gpu, _ = PT.run_gpu(w, plan=plan)
    assert gpu["status"] & 0x10
    assert (gpu["tiles_read"] == 0).all()
    plan.close()
    _check(w)


def test_cuda_graph_replay():
    import torch
    w = W.spec(groups=8)
    ref, plan = PT.run_gpu(w)
    d = PT.to_device(w)
    dev = torch.device("cuda", 0)
    out = dict(records=torch.full((w.rows, 258), PT.SENTINEL, dtype=torch.int32, device=dev),
               accepted=torch.zeros(w.groups, dtype=torch.int32, device=dev),
               emitted_tokens=torch.zeros(w.rows, dtype=torch.int32, device=dev),
               lse_out=torch.full((w.rows,), PT.LSE_SENTINEL, dtype=torch.float32, device=dev),
               status=torch.zeros(1, dtype=torch.int32, device=dev))
    plan.bind(**d, **out)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        plan.run(s)          # warm-up outside capture
        s.synchronize()
        with torch.cuda.graph(g, stream=s):
            plan.run(s)
    for _ in range(3):
        out["records"].fill_(PT.SENTINEL)
        g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(out["records"].cpu().numpy(), ref["records"])
    assert np.array_equal(out["emitted_tokens"].cpu().numpy(), ref["emitted_tokens"])
    plan.close()


def test_host_buffers_match_device_run():
    import torch
    w = W.spec(groups=4)
    ref, _ = PT.run_gpu(w)
    plan = PT.make_plan(w, host_staging=True)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
    arrays = dict(logits=pin(w.logits), group_indptr=pin(w.group_indptr), draft_tokens=pin(w.draft_tokens),
                  sampled_tokens=pin(w.sampled_tokens), requested=pin(w.requested), top_k=pin(w.top_k),
                  token_ids=pin(w.token_ids), id_counts=pin(w.id_counts),
                  records=pin(np.full((w.rows, 258), PT.SENTINEL, np.int32)),
                  accepted=pin(np.zeros(w.groups, np.int32)), emitted_tokens=pin(np.zeros(w.rows, np.int32)),
                  lse_out=pin(np.full(w.rows, PT.LSE_SENTINEL, np.float32)), status=pin(np.zeros(1, np.int32)))
    h2d, _ = plan.host_bytes(arrays)
    assert h2d < w.logits.nbytes // 2, "pinned logits are read in place, not copied"
    plan.run_host(arrays)
    torch.cuda.synchronize()
    assert np.array_equal(arrays["records"].numpy(), ref["records"])
    assert np.array_equal(arrays["accepted"].numpy(), ref["accepted"])
    assert np.array_equal(arrays["emitted_tokens"].numpy(), ref["emitted_tokens"])
    plan.close()


def test_host_buffers_pageable_logits_are_staged():
    # A logit block in ordinary (pageable) host memory is copied to device
    # staging; pinned blocks are read in place (the test above).  Same results.
    import torch
    w = W.large(groups=4)
    ref, _ = PT.run_gpu(w)
    plan = PT.make_plan(w, host_staging=True)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
    arrays = dict(logits=np.ascontiguousarray(w.logits), group_indptr=pin(w.group_indptr),
                  draft_tokens=pin(w.draft_tokens), sampled_tokens=pin(w.sampled_tokens),
                  requested=pin(w.requested), top_k=pin(w.top_k), token_ids=pin(w.token_ids),
                  id_counts=pin(w.id_counts), records=pin(np.full((w.rows, 258), PT.SENTINEL, np.int32)),
                  accepted=pin(np.zeros(w.groups, np.int32)), emitted_tokens=pin(np.zeros(w.rows, np.int32)),
                  lse_out=pin(np.full(w.rows, PT.LSE_SENTINEL, np.float32)), status=pin(np.zeros(1, np.int32)))
    h2d, _ = plan.host_bytes(arrays)
    assert h2d >= w.logits.nbytes, "pageable logits are copied whole"
    plan.run_host(arrays)
    torch.cuda.synchronize()
    assert np.array_equal(arrays["records"].numpy(), ref["records"])
    assert np.array_equal(arrays["accepted"].numpy(), ref["accepted"])
    assert np.array_equal(arrays["emitted_tokens"].numpy(), ref["emitted_tokens"])
    plan.close()


# ----------------------------------------------------------------- prompt scoring

def _score(w, targets, plan=None, **kw):
    gpu, plan = PT.run_gpu_score(w, targets, plan=plan, **kw)
    orc = PT.run_oracle_score(w, targets, THREADS)
    stats = PT.compare_score(w, targets, gpu, orc)
    te = PT.lpe_tile_elems(w.dtype)
    T = (w.V + te - 1) // te
    valid = (np.asarray(targets) >= 0) & (np.asarray(targets) < w.V)
    assert np.array_equal(gpu["tiles_read"], np.where(valid, T, 0)), "rows read: exactly the valid targets'"
    plan.close()
    return gpu, orc, stats


def _score_rows(rows_f32, V, *, dtype="f32", Vp=None):
    n = np.asarray(rows_f32).shape[0]
    return W.custom(rows_f32, V, [1] * n, dtype=dtype, Vp=Vp, k_max=0)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_score_prompt_workload(dtype):
    w = W.prompt(rows=48, dtype=dtype)
    _, _, st = _score(w, w.meta["targets"])
    assert st["scored"] >= 40 and st["ranks_above_1"] >= 20


def test_score_prompt_full_size():
    w = W.prompt()
    _, _, st = _score(w, w.meta["targets"])
    assert st["scored"] >= 480


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_score_collapse_rescans_every_tile(dtype):
    # one logit of 3e7, the others in [0, 0.5] over several tiles: every other
    # logprob rounds to the maximum's negated, so each non-maximal target has
    # rank 2 and every tile holds logits reported equal to the target's
    rng = np.random.default_rng(31)
    V = 40_000
    x = rng.uniform(0.0, 0.5, (6, V)).astype(np.float32)
    x[:, 17] = np.float32(3e7)
    targets = np.array([17, 0, V - 1, 20_000, 16_384, 8_191], np.int32)
    gpu, _, _ = _score(_score_rows(x, V, dtype=dtype), targets)
    assert gpu["records"][0][2] == 1 and (gpu["records"][1:, 2] == 2).all()


def test_score_fp32_subtraction_collisions():
    # FP32 logits near 0 under an lse near 1000: the ulp of the difference
    # (6e-5) merges many distinct logits with the target's
    rng = np.random.default_rng(32)
    V = 30_000
    x = rng.standard_normal((8, V)).astype(np.float32) * np.float32(1e-3)
    x[:, 5] = np.float32(1000.0)
    targets = np.array([0, 1, 2, 3, 4, 6, 29_999, 5], np.int32)
    gpu, _, _ = _score(_score_rows(x, V), targets)
    assert (gpu["records"][:7, 2] > 1).all() and gpu["records"][7][2] == 1


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_score_ties_invalid_and_masked(dtype):
    rng = np.random.default_rng(33)
    V = 20_000
    x = (np.round(rng.standard_normal((8, V)) * 4) / 4).astype(np.float32)
    x[2, ::3] = -np.inf                      # a masked vocabulary
    x[5, 1:] = -np.inf                       # a single live lane
    x[6, :100] = np.float32(-0.0)
    targets = np.array([int(np.argmax(x[0])), 7, 3, -1, V, 0, 50, V + 7], np.int32)
    gpu, orc, _ = _score(_score_rows(x, V, dtype=dtype), targets)
    assert gpu["status"] == 0x2
    assert gpu["records"][0][2] == 1
    assert gpu["records"][2][2] == 1 + int(np.isfinite(x[2]).sum())  # a masked target: below every live lane


@pytest.mark.parametrize("V,Vp,dtype", [(7, 8, "bf16"), (19, 20, "f32"), (1, 4, "f32"), (10_001, 10_008, "bf16"),
                                        (16_385, 16_388, "f32"), (8192, 8192, "f32")])
def test_score_ragged_vocabularies(V, Vp, dtype):
    rng = np.random.default_rng(V + 1)
    x = rng.normal(0, 2, (4, V)).astype(np.float32)
    targets = rng.integers(0, V, 4).astype(np.int32)
    _score(_score_rows(x, V, dtype=dtype, Vp=Vp), targets)


def test_score_and_generation_share_a_plan():
    # scoring on a plan between generation runs: poisoned scratch, no state left behind
    w = W.decode(rows=12)
    plan = PT.make_plan(w)
    _check(w, plan=plan, poison=True)
    plan = PT.make_plan(w)
    ws = W.prompt(rows=12)
    gpu, _ = PT.run_gpu_score(ws, ws.meta["targets"], plan=plan, poison=True)
    PT.compare_score(ws, ws.meta["targets"], gpu, PT.run_oracle_score(ws, ws.meta["targets"], THREADS))
    gen, _ = PT.run_gpu(w, plan=plan, poison=True)
    PT.compare(w, gen, PT.run_oracle(w, THREADS))
    plan.close()


def test_score_no_rows():
    w = W.prompt(rows=4)
    import torch
    import logprob_epilogue_gb300 as lpe
    plan = PT.make_plan(w)
    dev = torch.device("cuda", 0)
    st = torch.full((1,), -1, dtype=torch.int32, device=dev)
    plan.score(logits=torch.zeros((0, w.Vp), dtype=torch.bfloat16, device=dev),
               target_tokens=torch.zeros(1, dtype=torch.int32, device=dev),
               records=torch.zeros((1, lpe.SCORE_WORDS), dtype=torch.int32, device=dev), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    plan.close()


def _warp_share_ids(tile, V, dtype, warp):
    """Vocabulary ids of one compute warp's share of a 32 KiB tile (thread i reads
    the 16-byte vectors c*256 + i)."""
    epv = 8 if dtype == "bf16" else 4
    te = PT.lpe_tile_elems(dtype)
    tid = np.arange(32 * warp, 32 * warp + 32)
    c = np.arange(te // epv // 256)
    e = np.arange(epv)
    ids = ((c[:, None, None] * 256 + tid[None, :, None]) * epv + e[None, None, :]).reshape(-1)
    ids = tile * te + ids
    return ids[ids < V]


@pytest.mark.parametrize("dtype,ragged", [("bf16", False), ("bf16", True), ("f32", False), ("f32", True)])
def test_one_low_warp_forces_exact_select(dtype, ragged):
    # one warp's share of every tile far below the rest: the tile threshold (the
    # smallest warp's 4th-largest thread maximum) drops, so every other warp has
    # far more than 32 candidates and takes the exact per-warp selection
    te = PT.lpe_tile_elems(dtype)
    V = 3 * te + (777 if ragged else 0)
    rng = np.random.default_rng(41)
    x = rng.standard_normal((2, V)).astype(np.float32)
    for t in range((V + te - 1) // te):
        ids = _warp_share_ids(t, V, dtype, 7)
        x[:, ids] = np.float32(-10.0) + rng.standard_normal((2, ids.size)).astype(np.float32) * np.float32(0.01)
    x[1] = np.round(x[1] * 2) / 2  # heavy exact ties as well
    epv = 8 if dtype == "bf16" else 4
    Vp = (V + epv - 1) // epv * epv + (epv if ragged else 0)  # rows 16-byte aligned, plus one pad vector
    x0 = W.bf16_to_f32(W.bf16_bits(x[0])) if dtype == "bf16" else x[0]
    w = _one_group(x, V, dtype=dtype, Vp=Vp, k=1, drafts=[int(np.argmax(x0)), -1])
    gpu, _, _ = _check(w)
    assert gpu["accepted"].tolist() == [1]  # both rows carry records


# ----------------------------------------------------------------- commit clipping

@pytest.mark.parametrize("read_ahead", [False, True], ids=["prefix_only", "read_ahead"])
@pytest.mark.parametrize("name", ["spec", "large", "tiny"])
def test_commit_clipping(name, read_ahead):
    w = {"spec": lambda: W.spec(groups=16), "large": lambda: W.large(groups=12), "tiny": W.tiny}[name]()
    eos, budgets = W.commit_clip(w, 70 + len(name))
    plan = PT.make_plan(w, read_ahead=read_ahead)
    gpu, plan = PT.run_gpu(w, plan=plan, eos_tokens=eos, budgets=budgets)
    orc = PT.run_oracle(w, THREADS, eos_tokens=eos, budgets=budgets)
    PT.compare(w, gpu, orc)
    PT.check_tiles(w, orc, gpu["tiles_read"], strict=not read_ahead)
    assert (orc["accepted"] == -1).any() and (budgets <= 0).any()
    plan.close()


def test_commit_clipping_hand_checked_block():
    import oracle_pins as P
    w = P._clip_block()
    for eos, budgets in (([11, 11, 24, 99], None), (None, [2, 1, 0, 9]), ([7, 12, 22, -1], [3, 9, 9, 2])):
        e = None if eos is None else np.array(eos, np.int32)
        b = None if budgets is None else np.array(budgets, np.int32)
        gpu, plan = PT.run_gpu(w, eos_tokens=e, budgets=b)
        orc = PT.run_oracle(w, THREADS, eos_tokens=e, budgets=b)
        PT.compare(w, gpu, orc)
        PT.check_tiles(w, orc, gpu["tiles_read"], strict=True)
        plan.close()


def test_bind_clears_clipping():
    w = W.spec(groups=4, V=20_000, Vp=20_000)
    plan = PT.make_plan(w)
    PT.run_gpu(w, plan=plan, budgets=np.zeros(w.groups, np.int32))
    gpu, _ = PT.run_gpu(w, plan=plan)  # a new bind: unclipped
    PT.compare(w, gpu, PT.run_oracle(w, THREADS))
    plan.close()


def test_score_and_clip_argument_errors():
    # host-side checks only: each call returns before anything is enqueued
    import ctypes
    import torch
    import logprob_epilogue_gb300 as lpe
    L = lpe.lib()
    w = W.prompt(rows=4, V=1000, Vp=1000)
    plan = PT.make_plan(w, max_rows=4, max_groups=4)
    assert L.lp_bind_clip(plan._h, None, None) == -7          # nothing bound yet
    dev = torch.device("cuda", 0)
    buf = torch.zeros(64, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    io = lpe.ScoreIO(buf.data_ptr(), buf.data_ptr(), buf.data_ptr(), None, st.data_ptr(), 5)
    assert L.lp_score(plan._h, ctypes.byref(io), None) == -2   # rows > max_rows
    io = lpe.ScoreIO(buf.data_ptr() + 4, buf.data_ptr(), buf.data_ptr(), None, st.data_ptr(), 2)
    assert L.lp_score(plan._h, ctypes.byref(io), None) == -3   # logits not 16-byte aligned
    io = lpe.ScoreIO(None, buf.data_ptr(), buf.data_ptr(), None, st.data_ptr(), 2)
    assert L.lp_score(plan._h, ctypes.byref(io), None) == -1   # NULL logits
    plan.close()
    gpu, plan = PT.run_gpu(W.spec(groups=2, V=1000, Vp=1000), plan=PT.make_plan(W.spec(groups=2, V=1000, Vp=1000)))
    assert L.lp_bind_clip(plan._h, ctypes.c_void_p(buf.data_ptr() + 2), None) == -3  # misaligned
    plan.close()
