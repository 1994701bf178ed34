"""CPU checks of the C-ABI library: it builds, loads, exports every declared
symbol, and answers host-side calls without a GPU."""
import ctypes
import os
import re

import pytest

import logprob_epilogue_gb300 as lpe
from logprob_epilogue_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    B.build()
    return lpe.lib()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(lp_[a-z0-9_]+)\s*\(",
                                    text, re.M))
    return names


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 12
    for n in sorted(names):
        assert hasattr(L, n), n
    assert set(lpe.EXPORTS) == names


def test_strerror(L):
    for code in range(0, -8, -1):
        assert lpe.lib().lp_strerror(code)
    assert b"unknown" in lpe.lib().lp_strerror(-99)


def test_scratch_bytes_of_workloads(L):
    # tile partials dominate: per 32 KiB tile, one run-tagged (max, exp-sum)
    # pair and one prompt-scoring (count, minimum) per compute warp (8 x 16 and
    # 8 x 8 bytes) and 32 summary entries (256 bytes)
    b = lpe.scratch_bytes(max_rows=2048, max_groups=256, k_max=7, V=262_144, dtype="f32")
    assert 2048 * 32 * 448 <= b < 2048 * 32 * 448 + (1 << 20)
    assert lpe.scratch_bytes(max_rows=0, max_groups=1, k_max=0, V=10) == 0
    staged = lpe.scratch_bytes(max_rows=4, max_groups=1, k_max=3, V=1000, V_padded=1024, dtype="f32",
                               host_staging=True)
    assert staged > 4 * 1024 * 4


@pytest.mark.parametrize("kw,code", [
    (dict(max_rows=0), -2), (dict(V=100, V_padded=50), -2), (dict(k_max=16), -4), (dict(k_alt_max=33), -4),
    (dict(max_ids=129), -4), (dict(dtype="fp8"), -5), (dict(V=1001, V_padded=1001, dtype="bf16"), -3),
])
def test_create_rejects_bad_descriptors_before_any_cuda_call(L, kw, code):
    args = dict(max_rows=4, max_groups=2, k_max=3, V=1000, V_padded=1000, dtype="f32")
    args.update(kw)
    d = lpe.make_desc(**args)
    h = ctypes.c_void_p()
    assert L.lp_plan_create(ctypes.byref(h), ctypes.byref(d)) == code
    assert not h.value


def test_create_without_gpu_fails_cleanly(L):
    try:
        import torch
        if torch.cuda.is_available():
            pytest.skip("a GPU is present")
    except Exception:
        pass
    d = lpe.make_desc(max_rows=4, max_groups=2, k_max=3, V=1000, dtype="f32")
    h = ctypes.c_void_p()
    assert L.lp_plan_create(ctypes.byref(h), ctypes.byref(d)) == -6
    assert L.lp_last_cuda_error() != 0


def test_null_arguments(L):
    assert L.lp_bind(None, None) == -1
    assert L.lp_run(None, None) == -1
    assert L.lp_plan_destroy(None) == -1
    assert L.lp_plan_create(None, None) == -1
    assert L.lp_bind_clip(None, None, None) == -1
    assert L.lp_score(None, None, None) == -1


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(lpe, "_lib", None)
    monkeypatch.setattr(lpe, "LIB_PATH", str(tmp_path / "nope.so"))
    with pytest.raises(RuntimeError, match="missing"):
        lpe.lib()


def test_product_path_does_not_import_the_oracle():
    for dirpath, _, files in os.walk(os.path.join(ROOT, "logprob_epilogue_gb300")):
        for fn in files:
            if fn.endswith((".py", ".cu", ".h", ".cpp")):
                text = open(os.path.join(dirpath, fn)).read()
                assert "oracle" not in text.replace("the oracle", ""), fn
