"""lp_run_static, the entry point that allocates no device memory, against the
plan entry point (lp_plan_create + lp_bind + lp_run) on the same inputs.

Some callers cannot call cudaMalloc: a serving process whose framework has
reserved the whole device for its own caching allocator, code called back from
inside such an allocator, runtimes with a device-memory budget fixed at start.
lp_run_static gives them the same epilogue with its scratch in one fixed array
inside the library.  This file runs last so that a stop at its first failure
leaves every other test already run.
"""
import ctypes

import numpy as np
import pytest

import parity as PT
import workloads as W


def _desc(w):
    import logprob_epilogue_gb300 as lpe
    return lpe.make_desc(max_rows=max(w.rows, 1), max_groups=max(w.groups, 1), k_max=w.k_max, V=w.V,
                         V_padded=w.Vp, dtype=w.dtype, k_alt_max=20, max_ids=128, device=0)


def _run_static(w):
    """One lp_run_static call; outputs in the same form as PT.run_gpu's."""
    import torch
    import logprob_epilogue_gb300 as lpe
    dev = torch.device("cuda", 0)
    rows, G = w.rows, w.groups
    out = dict(
        records=torch.full((max(rows, 1), 258), PT.SENTINEL, dtype=torch.int32, device=dev),
        accepted=torch.full((max(G, 1),), -7, dtype=torch.int32, device=dev),
        emitted_tokens=torch.full((max(rows, 1),), -7, dtype=torch.int32, device=dev),
        lse_out=torch.full((max(rows, 1),), PT.LSE_SENTINEL, dtype=torch.float32, device=dev),
        status=torch.full((1,), -1, dtype=torch.int32, device=dev),
    )
    lpe.run_static(_desc(w), **PT.to_device(w), **out)
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy() for k, v in out.items()}
    res["records"] = res["records"][:rows]
    res["accepted"] = res["accepted"][:G]
    res["emitted_tokens"] = res["emitted_tokens"][:rows]
    res["lse"] = res["lse_out"][:rows]
    res["status"] = int(res["status"].view(np.uint32)[0])
    return res


def _same(w, static, planned):
    """Parity rule of the other GPU tests, with the plan entry point as the reference."""
    stats = PT.compare(w, static, planned, check_invariant=False)
    assert stats["rows_written"] > 0


@pytest.mark.gpu
def test_static_matches_plan_entry_point_two_calls():
    # Two calls in a row on different shapes and element types: the second
    # reuses the fixed array the first one left behind.
    first = W.spec()             # 512 rows x 248,448 BF16 lanes: about 3.7 MB of scratch
    second = W.large(groups=4)   # 32 rows x 262,144 FP32 lanes
    s1 = _run_static(first)
    s2 = _run_static(second)
    p1, plan1 = PT.run_gpu(first)
    plan1.close()
    p2, plan2 = PT.run_gpu(second)
    plan2.close()
    _same(first, s1, p1)
    _same(second, s2, p2)
    # and once more on the first input, after the second one's contents
    _same(first, _run_static(first), p1)


def test_static_rejects_runs_beyond_its_array():
    # No GPU needed: the size check comes before any CUDA call.  2,048 FP32
    # rows of 262,144 lanes need about 17 MB of scratch, above the 4 MiB array.
    import logprob_epilogue_gb300 as lpe
    try:
        L = lpe.lib()
    except (RuntimeError, OSError) as e:  # pragma: no cover - library not built
        pytest.skip(str(e))
    desc = lpe.make_desc(max_rows=2048, max_groups=256, k_max=7, V=262_144, dtype="f32")
    fake = 1 << 20  # aligned, never dereferenced
    io = lpe.IO(*([fake] * 11), None, fake, 2048, 256)
    rc = L.lp_run_static(ctypes.byref(desc), ctypes.byref(io), None)
    assert rc == -8, lpe.ERRORS.get(rc, rc)
    assert b"fixed array" in L.lp_strerror(-8)
    assert lpe.STATIC_SCRATCH_BYTES == 4 << 20
