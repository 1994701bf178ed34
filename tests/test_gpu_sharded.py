"""Vocabulary-sharded records (lp_run_sharded) against the unsharded oracle.

The records are built from per-shard exchanges (each shard's (max, exp-mass),
then its chosen raw logit and best 32 sort keys or selected-id raw logits), so
they must satisfy the same parity rule as lp_run's: bit-exact ids, logprobs
within the tolerance, near ties ordered consistently with the GPU's values.
"""
import os

import numpy as np
import pytest

import parity as PT
import workloads as W

pytestmark = pytest.mark.gpu
THREADS = os.cpu_count() or 8


def run_sharded(w, shards, plan=None):
    import torch
    if plan is None:
        plan = PT.make_plan(w, vocab_shards=True)
    dev = torch.device("cuda", 0)
    d = PT.to_device(w)
    rows, G = w.rows, w.groups
    out = dict(records=torch.full((max(rows, 1), 258), PT.SENTINEL, dtype=torch.int32, device=dev),
               accepted=torch.full((max(G, 1),), -7, dtype=torch.int32, device=dev),
               emitted_tokens=torch.full((max(rows, 1),), -7, dtype=torch.int32, device=dev),
               lse_out=torch.full((max(rows, 1),), PT.LSE_SENTINEL, dtype=torch.float32, device=dev),
               status=torch.full((1,), -1, dtype=torch.int32, device=dev))
    plan.bind(**d, **out)
    plan.run_sharded(shards)
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy() for k, v in out.items()}
    res["records"] = res["records"][:rows]
    res["accepted"] = res["accepted"][:G]
    res["emitted_tokens"] = res["emitted_tokens"][:rows]
    res["lse"] = res["lse_out"][:rows]
    res["status"] = int(res["status"].view(np.uint32)[0])
    res["tiles_read"] = plan.tiles_read(rows)
    return res, plan


def _check(w, shards):
    gpu, plan = run_sharded(w, shards)
    orc = PT.run_oracle(w, THREADS)
    stats = PT.compare(w, gpu, orc)
    PT.check_tiles(w, orc, gpu["tiles_read"], strict=True)
    plan.close()
    return stats


@pytest.mark.parametrize("shards", [2, 4, 8])
@pytest.mark.parametrize("name", ["spec", "large", "decode"])
def test_sharded_workloads(name, shards):
    w = {"spec": lambda: W.spec(groups=12), "large": lambda: W.large(groups=10),
         "decode": lambda: W.decode(rows=16)}[name]()
    stats = _check(w, shards)
    assert stats["rows_written"] > 0


@pytest.mark.parametrize("shards", [2, 8])
def test_sharded_full_size_spec(shards):
    assert _check(W.make("spec"), shards)["rows_written"] > 0


@pytest.mark.parametrize("shards", [3, 8])
def test_sharded_tie_across_shards(shards):
    # a 64-way exact tie at the maximum spread over every shard: the natural
    # list must be the 20 smallest tied ids, whichever shards hold them
    rng = np.random.default_rng(55)
    V = 8 * 16384 + 123
    x = rng.normal(0, 1, V).astype(np.float32)
    x[rng.choice(V, 64, replace=False)] = 16.0
    w = W.custom(x[None, :], V, [1], dtype="bf16", Vp=V + 5, k_max=0)
    _check(w, shards)


@pytest.mark.parametrize("shards", [2, 4])
def test_sharded_subtraction_ties(shards):
    # logits that collapse to one logprob after the subtraction, across shards
    rng = np.random.default_rng(56)
    V = 4 * 8192 + 77
    x = rng.uniform(0.0, 0.01, V).astype(np.float32)
    x[rng.integers(0, V)] = 1e4
    w = W.custom(np.stack([x, x[::-1].copy()]), V, [2], Vp=V + 3, k_max=1, drafts=[int(np.argmax(x)), -1])
    _check(w, shards)


def test_sharded_explicit_ids_and_errors():
    rng = np.random.default_rng(57)
    V = 5 * 8192
    x = rng.normal(0, 2, (3, V)).astype(np.float32)
    ids = [[0, V - 1, 8191, 8192, V + 4, -3, 3 * 8192 + 17], None, list(range(100, 228))]
    w = W.custom(x, V, [1, 1, 1], token_ids=ids, id_counts=[7, 0, 128], k_max=0)
    gpu, plan = run_sharded(w, 5)
    orc = PT.run_oracle(w, THREADS)
    PT.compare(w, gpu, orc)
    assert gpu["status"] & 0x1  # ids outside [0, V)
    plan.close()


def test_sharded_argument_errors():
    import logprob_epilogue_gb300 as lpe
    w = W.spec(groups=2)
    plain = PT.make_plan(w)
    with pytest.raises(lpe.LPError):  # no exchange buffers, and not bound
        plain.run_sharded(2)
    plain.close()
    gpu, plan = run_sharded(w, 2)
    T = plan.tiles_per_row
    for bad in (0, 9, T + 1):
        with pytest.raises(lpe.LPError):
            plan.run_sharded(bad)
    plan.close()
