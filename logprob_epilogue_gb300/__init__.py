"""Python binding of liblp_epilogue.so: the GB300 generation-logprob and greedy
speculative-acceptance epilogue.

Argument marshalling only: every step of the operation runs in the library's
CUDA kernels (see ``include/lp_epilogue.h`` for the contract).  PyTorch is used
for device memory and streams.  There is no fallback: if the library is not
built, or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "liblp_epilogue.so")

RECORD_WORDS = 258
SCORE_WORDS = 43  # prompt-scoring record: target id, lp bits, rank, 20 (id, lp bits) pairs
SCORE_ALTS = 20
MAX_IDS = 128
UNUSED_LP_BITS = 0x7FC00000
TILE_BYTES = 32768  # vocabulary tile: 16384 BF16 or 8192 FP32 logits

LP_F32, LP_BF16 = 0, 1
STATUS_BAD_ID = 0x1
STATUS_BAD_TOKEN = 0x2
STATUS_BAD_COUNT = 0x4
STATUS_BAD_GROUP = 0x8
STATUS_TIMEOUT = 0x10
PLAN_HOST_STAGING = 0x1
PLAN_READ_AHEAD = 0x2
PLAN_VOCAB_SHARDS = 0x4
PLAN_DEBUG_FORCE_TIMEOUT = 0x100
PLAN_DEBUG_TRACE = 0x200

ERRORS = {0: "LP_OK", -1: "LP_EINVAL", -2: "LP_ESHAPE", -3: "LP_EALIGN", -4: "LP_ECAPACITY",
          -5: "LP_EDTYPE", -6: "LP_ECUDA", -7: "LP_ESTATE", -8: "LP_ESCRATCH"}
STATIC_SCRATCH_BYTES = 4 << 20  # fixed device scratch of run_static

# Every symbol include/lp_epilogue.h declares.
EXPORTS = ("lp_plan_create", "lp_plan_destroy", "lp_plan_scratch_bytes", "lp_bind", "lp_run", "lp_run_host",
           "lp_run_host_bytes", "lp_debug_tiles_read", "lp_debug_poison_scratch", "lp_debug_trace",
           "lp_plan_tiles_per_row", "lp_run_static", "lp_score", "lp_bind_clip", "lp_debug_occupy",
           "lp_chain_verify", "lp_run_sharded",
           "lp_strerror", "lp_last_cuda_error")


class PlanDesc(ctypes.Structure):
    _fields_ = [
        ("max_rows", ctypes.c_int32),
        ("max_groups", ctypes.c_int32),
        ("k_max", ctypes.c_int32),
        ("V", ctypes.c_int64),
        ("V_padded", ctypes.c_int64),
        ("dtype", ctypes.c_int32),
        ("k_alt_max", ctypes.c_int32),
        ("max_ids", ctypes.c_int32),
        ("device", ctypes.c_int32),
        ("flags", ctypes.c_uint32),
        ("timeout_ns", ctypes.c_int64),
    ]


class IO(ctypes.Structure):
    _fields_ = [
        ("logits", ctypes.c_void_p),
        ("group_indptr", ctypes.c_void_p),
        ("draft_tokens", ctypes.c_void_p),
        ("sampled_tokens", ctypes.c_void_p),
        ("requested", ctypes.c_void_p),
        ("top_k", ctypes.c_void_p),
        ("token_ids", ctypes.c_void_p),
        ("id_counts", ctypes.c_void_p),
        ("records", ctypes.c_void_p),
        ("accepted", ctypes.c_void_p),
        ("emitted_tokens", ctypes.c_void_p),
        ("lse_out", ctypes.c_void_p),
        ("status", ctypes.c_void_p),
        ("rows", ctypes.c_int32),
        ("groups", ctypes.c_int32),
    ]


class ScoreIO(ctypes.Structure):
    _fields_ = [
        ("logits", ctypes.c_void_p),
        ("target_tokens", ctypes.c_void_p),
        ("records", ctypes.c_void_p),
        ("lse_out", ctypes.c_void_p),
        ("status", ctypes.c_void_p),
        ("rows", ctypes.c_int32),
    ]


class ChainIO(ctypes.Structure):
    _fields_ = [
        ("logits", ctypes.c_void_p),
        ("group_indptr", ctypes.c_void_p),
        ("draft_tokens", ctypes.c_void_p),
        ("draft_probs", ctypes.c_void_p),
        ("temperature", ctypes.c_void_p),
        ("u", ctypes.c_void_p),
        ("r", ctypes.c_void_p),
        ("accepted", ctypes.c_void_p),
        ("emitted", ctypes.c_void_p),
        ("lse_out", ctypes.c_void_p),
        ("status", ctypes.c_void_p),
        ("rows", ctypes.c_int32),
        ("groups", ctypes.c_int32),
    ]


_lib = None


class LPError(RuntimeError):
    def __init__(self, code: int, what: str):
        msg = lib().lp_strerror(code).decode() if _lib is not None else ""
        cuda = f" (cudaError {lib().lp_last_cuda_error()})" if code == -6 else ""
        super().__init__(f"{what}: {ERRORS.get(code, code)}: {msg}{cuda}")
        self.code = code


def lib() -> ctypes.CDLL:
    """Loads the in-tree library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with logprob_epilogue_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.c_void_p
        L.lp_plan_create.argtypes = [ctypes.POINTER(P), ctypes.POINTER(PlanDesc)]
        L.lp_plan_destroy.argtypes = [P]
        L.lp_plan_scratch_bytes.argtypes = [ctypes.POINTER(PlanDesc)]
        L.lp_plan_scratch_bytes.restype = ctypes.c_size_t
        L.lp_bind.argtypes = [P, ctypes.POINTER(IO)]
        L.lp_run.argtypes = [P, P]
        L.lp_run_host.argtypes = [P, ctypes.POINTER(IO), P]
        L.lp_run_host_bytes.argtypes = [P, ctypes.POINTER(IO), ctypes.POINTER(ctypes.c_int64),
                                        ctypes.POINTER(ctypes.c_int64)]
        L.lp_debug_tiles_read.argtypes = [P, P, ctypes.c_int32]
        L.lp_debug_poison_scratch.argtypes = [P, P]
        L.lp_plan_tiles_per_row.argtypes = [P]
        L.lp_debug_trace.argtypes = [P, P, P, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]
        L.lp_debug_occupy.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, P]
        L.lp_chain_verify.argtypes = [P, ctypes.POINTER(ChainIO), P]
        L.lp_run_sharded.argtypes = [P, ctypes.c_int32, P]
        L.lp_run_static.argtypes = [ctypes.POINTER(PlanDesc), ctypes.POINTER(IO), P]
        L.lp_score.argtypes = [P, ctypes.POINTER(ScoreIO), P]
        L.lp_bind_clip.argtypes = [P, P, P]
        L.lp_strerror.argtypes = [ctypes.c_int]
        L.lp_strerror.restype = ctypes.c_char_p
        L.lp_last_cuda_error.argtypes = []
        for name in EXPORTS:
            if name not in ("lp_plan_scratch_bytes", "lp_strerror"):
                getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise LPError(rc, what)


def make_desc(*, max_rows, max_groups, k_max, V, V_padded=None, dtype="bf16", k_alt_max=20, max_ids=128,
              device=0, host_staging=False, timeout_ns=0, debug_force_timeout=False, trace=False,
              read_ahead=False, vocab_shards=False) -> PlanDesc:
    flags = (PLAN_HOST_STAGING if host_staging else 0) | (PLAN_DEBUG_FORCE_TIMEOUT if debug_force_timeout else 0)
    flags |= (PLAN_DEBUG_TRACE if trace else 0) | (PLAN_READ_AHEAD if read_ahead else 0)
    flags |= PLAN_VOCAB_SHARDS if vocab_shards else 0
    return PlanDesc(int(max_rows), int(max_groups), int(k_max), int(V), int(V if V_padded is None else V_padded),
                    LP_BF16 if dtype == "bf16" else (LP_F32 if dtype == "f32" else 99), int(k_alt_max),
                    int(max_ids), int(device), flags, int(timeout_ns))


def scratch_bytes(**desc_kw) -> int:
    d = make_desc(**desc_kw)
    return int(lib().lp_plan_scratch_bytes(ctypes.byref(d)))


_IO_NAMES = ("logits", "group_indptr", "draft_tokens", "sampled_tokens", "requested", "top_k", "token_ids",
             "id_counts", "records", "accepted", "emitted_tokens", "lse_out", "status")


class Plan:
    """One epilogue plan (device scratch allocated once at creation)."""

    def __init__(self, **desc_kw):
        self.desc = make_desc(**desc_kw)
        self.dtype = desc_kw.get("dtype", "bf16")
        self.device = int(desc_kw.get("device", 0))
        h = ctypes.c_void_p()
        _check(lib().lp_plan_create(ctypes.byref(h), ctypes.byref(self.desc)), "lp_plan_create")
        self._h = h
        self._keep = None
        self.rows = 0
        self.groups = 0

    @property
    def tiles_per_row(self) -> int:
        return int(lib().lp_plan_tiles_per_row(self._h))

    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            _check(lib().lp_plan_destroy(self._h), "lp_plan_destroy")
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _io(self, tensors: dict, rows: int, groups: int, ptr) -> IO:
        vals = [ptr(tensors.get(n)) for n in _IO_NAMES]
        return IO(*vals, int(rows), int(groups))

    def bind(self, *, logits, group_indptr, draft_tokens, sampled_tokens, requested, top_k, token_ids,
             id_counts, records, accepted, emitted_tokens, status, lse_out=None) -> None:
        """Binds CUDA tensors (contiguous; int32 except logits, lse_out and status)."""
        import torch
        t = dict(logits=logits, group_indptr=group_indptr, draft_tokens=draft_tokens,
                 sampled_tokens=sampled_tokens, requested=requested, top_k=top_k, token_ids=token_ids,
                 id_counts=id_counts, records=records, accepted=accepted, emitted_tokens=emitted_tokens,
                 status=status, lse_out=lse_out)
        want_logit = torch.bfloat16 if self.dtype == "bf16" else torch.float32
        for name, x in t.items():
            if x is None:
                continue
            if not isinstance(x, torch.Tensor) or not x.is_cuda or x.device.index != self.device:
                raise ValueError(f"{name}: expected a CUDA tensor on device {self.device}")
            if not x.is_contiguous():
                raise ValueError(f"{name}: must be contiguous")
            if name == "logits":
                if x.dtype != want_logit or x.dim() != 2 or x.shape[1] != self.desc.V_padded:
                    raise ValueError(f"logits: expected {want_logit} [rows, {self.desc.V_padded}]")
            elif name == "lse_out":
                if x.dtype != torch.float32:
                    raise ValueError("lse_out: expected float32")
            elif name == "status":
                if x.element_size() != 4 or x.numel() < 1:
                    raise ValueError("status: expected one 32-bit word")
            elif x.dtype != torch.int32:
                raise ValueError(f"{name}: expected int32")
        rows = int(logits.shape[0])
        groups = int(group_indptr.numel()) - 1
        if records.numel() < rows * RECORD_WORDS or emitted_tokens.numel() < rows or draft_tokens.numel() < rows:
            raise ValueError("records / emitted_tokens / draft_tokens smaller than rows")
        for name in ("sampled_tokens", "requested", "top_k", "id_counts", "accepted"):
            if t[name].numel() < groups:
                raise ValueError(f"{name} smaller than groups")
        if token_ids.numel() < groups * MAX_IDS:
            raise ValueError("token_ids smaller than groups * 128")
        if lse_out is not None and lse_out.numel() < rows:
            raise ValueError("lse_out smaller than rows")
        io = self._io(t, rows, groups, lambda x: None if x is None else x.data_ptr())
        _check(lib().lp_bind(self._h, ctypes.byref(io)), "lp_bind")
        self._keep = t
        self.rows, self.groups = rows, groups

    def bind_clip(self, *, eos_tokens=None, budgets=None) -> None:
        """Attaches per-group commit clipping (int32 CUDA tensors of [groups], or
        None) to the bound buffers for the following runs: the emitted prefix
        ends at an emitted EOS token (kept) and holds at most ``budgets[g]``
        tokens (<= 0: the group takes no step).  ``bind`` clears it."""
        import torch
        for name, x in (("eos_tokens", eos_tokens), ("budgets", budgets)):
            if x is None:
                continue
            if not isinstance(x, torch.Tensor) or not x.is_cuda or x.device.index != self.device:
                raise ValueError(f"{name}: expected a CUDA tensor on device {self.device}")
            if x.dtype != torch.int32 or not x.is_contiguous() or x.numel() < self.groups:
                raise ValueError(f"{name}: expected contiguous int32 [groups]")
        ptr = lambda x: None if x is None else x.data_ptr()  # noqa: E731
        _check(lib().lp_bind_clip(self._h, ptr(eos_tokens), ptr(budgets)), "lp_bind_clip")
        self._keep_clip = (eos_tokens, budgets)

    def run(self, stream=None) -> None:
        """Enqueues the epilogue on ``stream`` (default: torch's current stream)."""
        import torch
        if stream is None:
            stream = torch.cuda.current_stream(self.device)
        handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        _check(lib().lp_run(self._h, ctypes.c_void_p(handle)), "lp_run")

    def run_sharded(self, shards: int, stream=None) -> None:
        """Enqueues the bound epilogue with the records built over ``shards``
        vocabulary shards (plan created with ``vocab_shards=True``)."""
        import torch
        if stream is None:
            stream = torch.cuda.current_stream(self.device)
        handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        _check(lib().lp_run_sharded(self._h, int(shards), ctypes.c_void_p(handle)), "lp_run_sharded")

    def score(self, *, logits, target_tokens, records, status, lse_out=None, stream=None) -> None:
        """Enqueues prompt scoring of ``target_tokens`` (int32 [rows]) against
        ``logits`` [rows, V_padded]: ``records`` (int32 [rows, 43]) receives per row
        the target id, the FP32 bits of its logprob, its rank and the 20 natural
        alternatives; an invalid target (-1, or >= V) gives the invalid record.
        The bound tensors are not used."""
        import torch
        want_logit = torch.bfloat16 if self.dtype == "bf16" else torch.float32
        t = dict(logits=logits, target_tokens=target_tokens, records=records, status=status, lse_out=lse_out)
        for name, x in t.items():
            if x is None:
                continue
            if not isinstance(x, torch.Tensor) or not x.is_cuda or x.device.index != self.device:
                raise ValueError(f"{name}: expected a CUDA tensor on device {self.device}")
            if not x.is_contiguous():
                raise ValueError(f"{name}: must be contiguous")
        if logits.dtype != want_logit or logits.dim() != 2 or logits.shape[1] != self.desc.V_padded:
            raise ValueError(f"logits: expected {want_logit} [rows, {self.desc.V_padded}]")
        rows = int(logits.shape[0])
        if target_tokens.dtype != torch.int32 or target_tokens.numel() < rows:
            raise ValueError("target_tokens: expected int32 [rows]")
        if records.dtype != torch.int32 or records.numel() < rows * SCORE_WORDS:
            raise ValueError("records: expected int32 [rows, 43]")
        if status.element_size() != 4 or status.numel() < 1:
            raise ValueError("status: expected one 32-bit word")
        if lse_out is not None and (lse_out.dtype != torch.float32 or lse_out.numel() < rows):
            raise ValueError("lse_out: expected float32 [rows]")
        io = ScoreIO(logits.data_ptr(), target_tokens.data_ptr(), records.data_ptr(),
                     None if lse_out is None else lse_out.data_ptr(), status.data_ptr(), rows)
        if stream is None:
            stream = torch.cuda.current_stream(self.device)
        handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        self._keep_score = t
        _check(lib().lp_score(self._h, ctypes.byref(io), ctypes.c_void_p(handle)), "lp_score")

    def chain_verify(self, *, logits, group_indptr, draft_tokens, draft_probs, temperature, u, r, accepted,
                     emitted, status, lse_out=None, stream=None) -> None:
        """Enqueues stochastic chain verification: for each group, drafts
        accepted with probability min(1, p/q), the residual or bonus token drawn
        with the group's uniform r.  ``draft_probs`` is float32 [rows, V_padded]
        (the law that drew each draft), ``temperature`` and ``r`` float32
        [groups], ``u`` float32 [rows]; outputs ``accepted`` int32 [groups],
        ``emitted`` int32 [rows], optional ``lse_out`` float32 [rows] (lse of
        x / t).  The bound tensors are not used."""
        import torch
        want_logit = torch.bfloat16 if self.dtype == "bf16" else torch.float32
        t = dict(logits=logits, group_indptr=group_indptr, draft_tokens=draft_tokens, draft_probs=draft_probs,
                 temperature=temperature, u=u, r=r, accepted=accepted, emitted=emitted, status=status,
                 lse_out=lse_out)
        for name, x in t.items():
            if x is None:
                continue
            if not isinstance(x, torch.Tensor) or not x.is_cuda or x.device.index != self.device:
                raise ValueError(f"{name}: expected a CUDA tensor on device {self.device}")
            if not x.is_contiguous():
                raise ValueError(f"{name}: must be contiguous")
        if logits.dtype != want_logit or logits.dim() != 2 or logits.shape[1] != self.desc.V_padded:
            raise ValueError(f"logits: expected {want_logit} [rows, {self.desc.V_padded}]")
        rows, groups = int(logits.shape[0]), int(group_indptr.numel()) - 1
        if draft_probs.dtype != torch.float32 or tuple(draft_probs.shape) != tuple(logits.shape):
            raise ValueError("draft_probs: expected float32 of the logits' shape")
        for name in ("group_indptr", "draft_tokens", "accepted", "emitted"):
            if t[name].dtype != torch.int32:
                raise ValueError(f"{name}: expected int32")
        for name in ("temperature", "u", "r"):
            if t[name].dtype != torch.float32:
                raise ValueError(f"{name}: expected float32")
        if draft_tokens.numel() < rows or u.numel() < rows or emitted.numel() < rows:
            raise ValueError("draft_tokens, u, emitted: expected [rows]")
        if temperature.numel() < groups or r.numel() < groups or accepted.numel() < groups:
            raise ValueError("temperature, r, accepted: expected [groups]")
        io = ChainIO(logits.data_ptr(), group_indptr.data_ptr(), draft_tokens.data_ptr(), draft_probs.data_ptr(),
                     temperature.data_ptr(), u.data_ptr(), r.data_ptr(), accepted.data_ptr(), emitted.data_ptr(),
                     None if lse_out is None else lse_out.data_ptr(), status.data_ptr(), rows, groups)
        if stream is None:
            stream = torch.cuda.current_stream(self.device)
        handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        self._keep_chain = t
        _check(lib().lp_chain_verify(self._h, ctypes.byref(io), ctypes.c_void_p(handle)), "lp_chain_verify")

    def host_io(self, arrays: dict) -> IO:
        rows = int(arrays["logits"].shape[0])
        groups = int(np.asarray(arrays["group_indptr"]).size) - 1

        def ptr(a):
            if a is None:
                return None
            if hasattr(a, "data_ptr"):
                return a.data_ptr()
            return a.ctypes.data
        return self._io(arrays, rows, groups, ptr)

    def run_host(self, arrays: dict, stream=None) -> None:
        """Runs over host arrays (numpy or pinned CPU tensors); outputs land in the
        output arrays once ``stream`` is synchronised."""
        import torch
        io = self.host_io(arrays)
        if stream is None:
            stream = torch.cuda.current_stream(self.device)
        handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        self._keep_host = (arrays, io)
        _check(lib().lp_run_host(self._h, ctypes.byref(io), ctypes.c_void_p(handle)), "lp_run_host")

    def host_bytes(self, arrays: dict):
        io = self.host_io(arrays)
        h2d, d2h = ctypes.c_int64(), ctypes.c_int64()
        _check(lib().lp_run_host_bytes(self._h, ctypes.byref(io), ctypes.byref(h2d), ctypes.byref(d2h)),
               "lp_run_host_bytes")
        return int(h2d.value), int(d2h.value)

    def tiles_read(self, rows: int | None = None) -> np.ndarray:
        """Tiles the last run read per row (synchronises the last stream)."""
        rows = self.rows if rows is None else rows
        out = np.zeros(max(rows, 1), np.int32)
        _check(lib().lp_debug_tiles_read(self._h, out.ctypes.data, int(rows)), "lp_debug_tiles_read")
        return out[:rows]

    def trace(self):
        """Device timeline of the last run: (events uint64 [ctas*4+1, cap, 2], counts uint32 [ctas, 4]).

        Rings per CTA: producer, compute, merge (decisions), record kernel.  Event word 1 =
        type << 56 | row << 24 | tile (types: 1 kernel start, 2 claim, 3 TMA issue, 4 tile start,
        5 tile end, 6 tile published, 7 merge start, 8 acceptance decided, 9 merge end, 10/11
        prepare start/end, 12 producer exit, 17/18 record start/end, 19-21 record phases)."""
        ctas, cap = ctypes.c_int32(), ctypes.c_int32()
        _check(lib().lp_debug_trace(self._h, None, None, ctypes.byref(ctas), ctypes.byref(cap)), "lp_debug_trace")
        ev = np.zeros(((ctas.value * 4 + 1), cap.value, 2), np.uint64)
        cnt = np.zeros((ctas.value, 4), np.uint32)
        _check(lib().lp_debug_trace(self._h, ev.ctypes.data, cnt.ctypes.data, ctypes.byref(ctas), ctypes.byref(cap)),
               "lp_debug_trace")
        return ev, cnt

    def poison_scratch(self, stream=None) -> None:
        import torch
        if stream is None:
            stream = torch.cuda.current_stream(self.device)
        _check(lib().lp_debug_poison_scratch(self._h, ctypes.c_void_p(stream.cuda_stream)), "lp_debug_poison_scratch")


def debug_occupy(device: int, ctas: int, ns: int, stream) -> None:
    """Test hook: ``ctas`` CTAs on ``stream`` that each hold a multiprocessor's
    shared memory and spin for ``ns`` nanoseconds."""
    _check(lib().lp_debug_occupy(int(device), int(ctas), int(ns), ctypes.c_void_p(stream.cuda_stream)),
           "lp_debug_occupy")


def run_static(desc: PlanDesc, *, logits, group_indptr, draft_tokens, sampled_tokens, requested, top_k,
               token_ids, id_counts, records, accepted, emitted_tokens, status, lse_out=None, stream=None) -> None:
    """Enqueues the epilogue through ``lp_run_static``: the same operation as
    ``Plan(...).bind(...); run()``, but with no device allocation at all.

    For callers that may not allocate device memory (a framework whose caching
    allocator already holds the device, code called back from inside such an
    allocator, runtimes with a fixed memory budget).  The scratch is one fixed
    array of ``STATIC_SCRATCH_BYTES`` inside the library, shared by every call:
    runs that need more are refused with ``LP_ESCRATCH``, and calls that can
    overlap on the GPU (different streams or threads) race; keep them on one
    stream.  The first call on a device sets it up; make it before any stream
    capture on that device.  Buffers are CUDA tensors as for ``Plan.bind``."""
    import torch
    t = dict(logits=logits, group_indptr=group_indptr, draft_tokens=draft_tokens, sampled_tokens=sampled_tokens,
             requested=requested, top_k=top_k, token_ids=token_ids, id_counts=id_counts, records=records,
             accepted=accepted, emitted_tokens=emitted_tokens, status=status, lse_out=lse_out)
    for name, x in t.items():
        if x is None:
            continue
        if not isinstance(x, torch.Tensor) or not x.is_cuda or not x.is_contiguous():
            raise ValueError(f"{name}: expected a contiguous CUDA tensor")
    rows = int(logits.shape[0])
    groups = int(group_indptr.numel()) - 1
    io = IO(*[None if t[n] is None else t[n].data_ptr() for n in _IO_NAMES], rows, groups)
    if stream is None:
        stream = torch.cuda.current_stream(logits.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    _check(lib().lp_run_static(ctypes.byref(desc), ctypes.byref(io), ctypes.c_void_p(handle)), "lp_run_static")
