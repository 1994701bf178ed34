"""Plain CPU oracle for the logprob / greedy-acceptance epilogue.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
(``logprob_epilogue_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``lp_oracle.cpp`` (plain C++, FP64 logsumexp rounded to
FP32, FP32 subtraction, full stable sort per row); this module only builds that
file with g++ and marshals numpy arrays through ctypes.

Sources: "logprobs-design.md" (generation-logprob contract: definition of the
logprob, alternative ordering, explicit ids, packed record) and "mtp-design.md"
("A speculative round is a state transaction", verify and accept steps).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lp_oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "liblp_oracle.so")

RECORD_WORDS = 258
MAX_PAIRS = 128
NAN_BITS = 0x7FC00000
STATUS_BAD_ID = 0x1
STATUS_BAD_TOKEN = 0x2
STATUS_BAD_COUNT = 0x4
STATUS_BAD_GROUP = 0x8
SCORE_WORDS = 43
SCORE_ALTS = 20

_default = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile an oracle source (default: lp_oracle.cpp) into a shared library with g++."""
    hdr = os.path.join(_HERE, "lp_oracle.h")
    if force or not os.path.exists(out) or os.path.getmtime(out) < max(
        os.path.getmtime(src), os.path.getmtime(hdr)
    ):
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
               "-I", _HERE, "-o", tmp, src]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


class _IO(ctypes.Structure):
    _fields_ = [
        ("logits", ctypes.c_void_p),
        ("rows", ctypes.c_int64),
        ("V", ctypes.c_int64),
        ("Vp", ctypes.c_int64),
        ("groups", ctypes.c_int32),
        ("group_indptr", ctypes.c_void_p),
        ("draft_tokens", ctypes.c_void_p),
        ("sampled_tokens", ctypes.c_void_p),
        ("requested", ctypes.c_void_p),
        ("top_k", ctypes.c_void_p),
        ("token_ids", ctypes.c_void_p),
        ("id_counts", ctypes.c_void_p),
        ("k_max", ctypes.c_int32),
        ("k_alt_max", ctypes.c_int32),
        ("max_ids", ctypes.c_int32),
        ("records", ctypes.c_void_p),
        ("accepted", ctypes.c_void_p),
        ("emitted_tokens", ctypes.c_void_p),
        ("lse_out", ctypes.c_void_p),
        ("status", ctypes.c_void_p),
        ("rows_read", ctypes.c_void_p),
        ("eos_tokens", ctypes.c_void_p),
        ("budgets", ctypes.c_void_p),
    ]


def _f32(x) -> np.ndarray:
    a = np.ascontiguousarray(x, dtype=np.float32)
    if a.ndim != 1:
        a = a.reshape(-1)
    return a


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: str):
        L = ctypes.CDLL(path)
        L.orc_lse.restype = ctypes.c_float
        L.orc_lse.argtypes = [ctypes.c_void_p, ctypes.c_int64]
        L.orc_argmax.restype = ctypes.c_int32
        L.orc_argmax.argtypes = [ctypes.c_void_p, ctypes.c_int64]
        L.orc_logprob.restype = ctypes.c_float
        L.orc_logprob.argtypes = [ctypes.c_float, ctypes.c_float]
        L.orc_topk.restype = ctypes.c_int32
        L.orc_topk.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int32,
                               ctypes.c_void_p, ctypes.c_void_p]
        L.orc_epilogue.restype = ctypes.c_int
        L.orc_epilogue.argtypes = [ctypes.POINTER(_IO), ctypes.c_int]
        L.orc_rank.restype = ctypes.c_int32
        L.orc_rank.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_float]
        L.orc_chain_verify.restype = ctypes.c_int
        L.orc_chain_verify.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                       ctypes.c_int32] + [ctypes.c_void_p] * 8
        L.orc_score.restype = ctypes.c_int
        L.orc_score.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        self.L = L
        self.path = path

    def lse(self, x) -> np.float32:
        """FP64 logsumexp of a 1-D row, rounded to FP32."""
        a = _f32(x)
        return np.float32(self.L.orc_lse(_ptr(a), a.size))

    def argmax(self, x) -> int:
        """Smallest index among the maximal raw logits (-0 == +0)."""
        a = _f32(x)
        return int(self.L.orc_argmax(_ptr(a), a.size))

    def logprob(self, x, lse_value) -> np.float32:
        """fl32(x - lse) with -0 reported as +0."""
        return np.float32(self.L.orc_logprob(float(np.float32(x)), float(np.float32(lse_value))))

    def topk(self, x, K: int, lse_value=None):
        """Natural alternatives of a row: (ids int32[n], lps float32[n]), n = min(K, V)."""
        a = _f32(x)
        if lse_value is None:
            lse_value = self.lse(a)
        ids = np.full(max(K, 1), -1, np.int32)
        lps = np.zeros(max(K, 1), np.float32)
        n = self.L.orc_topk(_ptr(a), a.size, float(np.float32(lse_value)), int(K), _ptr(ids), _ptr(lps))
        return ids[:n].copy(), lps[:n].copy()

    def epilogue(self, *args, **kw):
        return _epilogue(self.L, *args, **kw)

    def rank(self, x, lse_value, lp) -> int:
        """1 + the number of lanes whose reported logprob is strictly greater than lp."""
        a = _f32(x)
        return int(self.L.orc_rank(_ptr(a), a.size, float(np.float32(lse_value)), float(np.float32(lp))))

    def score(self, logits: np.ndarray, V: int, targets, *, records=None, threads: int = 1):
        """Prompt scoring of float32 rows [rows, Vp]: dict of records [rows, 43], lse (NaN for
        invalid rows) and status."""
        logits = np.ascontiguousarray(logits, dtype=np.float32)
        rows, Vp = logits.shape
        tg = np.ascontiguousarray(targets, np.int32)
        if records is None:
            records = np.zeros((rows, SCORE_WORDS), np.int32)
        records = np.ascontiguousarray(records, np.int32)
        lse_out = np.full(max(rows, 1), np.nan, np.float32)
        status = np.zeros(1, np.uint32)
        rc = self.L.orc_score(_ptr(logits), rows, int(V), Vp, _ptr(tg), _ptr(records), _ptr(lse_out), _ptr(status),
                              int(threads))
        if rc != 0:
            raise RuntimeError(f"orc_score failed: {rc}")
        return {"records": records, "lse": lse_out[:rows], "status": int(status[0])}

    def chain_verify(self, logits: np.ndarray, V: int, group_indptr, draft_tokens, draft_probs, temperature,
                     u, r):
        """Stochastic chain verification of float32 rows [rows, Vp] with draft laws
        draft_probs [rows, Vp] and the uniforms u [rows], r [groups]: dict of
        accepted [groups] and emitted_tokens [rows]."""
        logits = np.ascontiguousarray(logits, dtype=np.float32)
        rows, Vp = logits.shape
        q = np.ascontiguousarray(draft_probs, np.float32)
        assert q.shape == logits.shape
        ip = np.ascontiguousarray(group_indptr, np.int32)
        G = ip.size - 1
        dr = np.ascontiguousarray(draft_tokens, np.int32)
        tt = np.ascontiguousarray(temperature, np.float32)
        uu = np.ascontiguousarray(u, np.float32)
        rr = np.ascontiguousarray(r, np.float32)
        accepted = np.full(max(G, 1), -7, np.int32)
        emitted = np.full(max(rows, 1), -7, np.int32)
        rc = self.L.orc_chain_verify(_ptr(logits), rows, int(V), Vp, G, _ptr(ip), _ptr(dr), _ptr(q), _ptr(tt),
                                     _ptr(uu), _ptr(rr), _ptr(accepted), _ptr(emitted))
        if rc != 0:
            raise RuntimeError(f"orc_chain_verify failed: {rc}")
        return {"accepted": accepted[:G], "emitted_tokens": emitted[:rows]}


def load(path: str | None = None) -> Oracle:
    """The default oracle (built on first use), or the library at ``path``."""
    global _default
    if path is not None:
        return Oracle(path)
    if _default is None:
        _default = Oracle(build())
    return _default


def lse(x):
    return load().lse(x)


def argmax(x):
    return load().argmax(x)


def logprob(x, lse_value):
    return load().logprob(x, lse_value)


def topk(x, K, lse_value=None):
    return load().topk(x, K, lse_value)


def epilogue(*args, **kw):
    return load().epilogue(*args, **kw)


def rank(x, lse_value, lp):
    return load().rank(x, lse_value, lp)


def score(*args, **kw):
    return load().score(*args, **kw)


def chain_verify(*args, **kw):
    return load().chain_verify(*args, **kw)


def _epilogue(L, logits: np.ndarray, V: int, group_indptr, draft_tokens, sampled_tokens, requested,
             top_k, token_ids, id_counts, *, k_max: int = 15, k_alt_max: int = 20,
             max_ids: int = 128, records=None, threads: int = 1, eos_tokens=None, budgets=None):
    """Runs the whole epilogue on host arrays.

    ``logits`` is float32 [rows, Vp] (BF16 data widened exactly).  ``records``
    may be passed pre-filled (e.g. with a sentinel) to check that rows not
    emitted are left untouched.  Returns a dict with records, accepted,
    emitted_tokens, lse (NaN where not computed), status and rows_read.
    ``eos_tokens`` and ``budgets`` ([groups] each, optional) clip the emitted
    prefix.
    """
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    rows, Vp = logits.shape
    G = len(group_indptr) - 1
    ip = np.ascontiguousarray(group_indptr, np.int32)
    dr = np.ascontiguousarray(draft_tokens, np.int32)
    sa = np.ascontiguousarray(sampled_tokens, np.int32)
    rq = np.ascontiguousarray(requested, np.int32)
    tk = np.ascontiguousarray(top_k, np.int32)
    ti = np.ascontiguousarray(token_ids, np.int32).reshape(G, MAX_PAIRS) if G > 0 else np.zeros((0, MAX_PAIRS), np.int32)
    ic = np.ascontiguousarray(id_counts, np.int32)
    if records is None:
        records = np.zeros((rows, RECORD_WORDS), np.int32)
    records = np.ascontiguousarray(records, np.int32)
    accepted = np.full(max(G, 1), -7, np.int32)
    emitted = np.full(max(rows, 1), -7, np.int32)
    lse_out = np.full(max(rows, 1), np.nan, np.float32)
    status = np.zeros(1, np.uint32)
    rows_read = np.zeros(1, np.int64)
    eo = None if eos_tokens is None else np.ascontiguousarray(eos_tokens, np.int32)
    bu = None if budgets is None else np.ascontiguousarray(budgets, np.int32)
    io = _IO(
        _ptr(logits), rows, int(V), Vp, G, _ptr(ip), _ptr(dr), _ptr(sa), _ptr(rq), _ptr(tk),
        _ptr(ti), _ptr(ic), int(k_max), int(k_alt_max), int(max_ids), _ptr(records), _ptr(accepted),
        _ptr(emitted), _ptr(lse_out), _ptr(status), _ptr(rows_read),
        None if eo is None else _ptr(eo), None if bu is None else _ptr(bu),
    )
    rc = L.orc_epilogue(ctypes.byref(io), int(threads))
    if rc != 0:
        raise RuntimeError(f"orc_epilogue failed: {rc}")
    return {
        "records": records,
        "accepted": accepted[:G],
        "emitted_tokens": emitted[:rows],
        "lse": lse_out[:rows],
        "status": int(status[0]),
        "rows_read": int(rows_read[0]),
    }
