"""Seeded synthetic inputs for the logprob / greedy-acceptance epilogue.

This module only draws inputs; it holds none of the epilogue's arithmetic (no
logsumexp, logprob, ordering or acceptance).  Both the CUDA path and the CPU
oracle consume the arrays it returns; neither imports the other.

Five workloads, with the shapes and value distributions of the epilogue's
target cases (verify groups of k drafts + 1 target row; requests asking for
K natural alternatives or up to 128 explicit ids):

  tiny   6 x 1,000 (row stride 1,024) FP32, round(N(0,2)*8)/8, 5% of lanes +-0
  decode 64 x 151,936 (stride 152,064) BF16, N(0,2.5) + 3 spikes of +U[12,18]
  spec   512 x 248,320 (stride 248,448) BF16, N(0,3), 128 groups of k=3
  large  2,048 x 262,144 FP32 holding BF16-rounded N(0,4), 256 groups of k=7
  wide   4 x 1,048,576 (stride 1,048,704) BF16, N(0,1), 1% of lanes +8,
         a 64-way exact tie at the maximum, one group of k=3

and, for prompt scoring, one target token per row:

  prompt 512 x 151,936 (stride 152,064) BF16, N(0,2.5) + 3 spikes, targets
         30% spike ids, 3% -1, the rest uniform

Pad lanes (between V and the row stride) hold +1e30 so that any leak into a
result is visible.  Where a draft must equal its row's argmax, the generator
plants that argmax: it writes a value above every other lane of the row (the
row maximum + a step that is exact in the element type) at a seed-drawn id,
or, in the wide workload, a tie group whose smallest id is the draft.  A
draft that must not match is a seed-drawn id different from the planted one.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

MAX_IDS = 128
PAD_VALUE = 1e30

SEEDS = {"tiny": 0, "decode": 1, "spec": 2, "large": 3, "wide": 4, "prompt": 5}
NAMES = ("tiny", "decode", "spec", "large", "wide")


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to BF16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (r >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of BF16 bits to float32."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass
class Workload:
    name: str
    dtype: str                 # "f32" or "bf16"
    V: int
    Vp: int
    k_max: int
    logits: np.ndarray         # [rows, Vp]: float32, or uint16 BF16 bits
    group_indptr: np.ndarray   # int32 [G+1]
    draft_tokens: np.ndarray   # int32 [rows]
    sampled_tokens: np.ndarray  # int32 [G]
    requested: np.ndarray      # int32 [G]
    top_k: np.ndarray          # int32 [G]
    token_ids: np.ndarray      # int32 [G, 128]
    id_counts: np.ndarray      # int32 [G]
    planted_argmax: np.ndarray  # int32 [rows]; -1 where nothing was planted
    meta: dict = field(default_factory=dict)

    @property
    def rows(self) -> int:
        return int(self.logits.shape[0])

    @property
    def groups(self) -> int:
        return int(self.group_indptr.shape[0] - 1)

    @property
    def elt(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def logits_f32(self, rows=None) -> np.ndarray:
        """Rows of the block as float32 (BF16 widened exactly)."""
        src = self.logits if rows is None else self.logits[rows]
        if self.dtype == "bf16":
            return bf16_to_f32(src)
        return np.ascontiguousarray(src, dtype=np.float32)

    def inputs(self) -> dict:
        return dict(group_indptr=self.group_indptr, draft_tokens=self.draft_tokens,
                    sampled_tokens=self.sampled_tokens, requested=self.requested,
                    top_k=self.top_k, token_ids=self.token_ids, id_counts=self.id_counts)


def _distinct_ids(rng, V: int, n: int, exclude=()) -> np.ndarray:
    ex = set(int(e) for e in exclude)
    out: list[int] = []
    seen = set(ex)
    while len(out) < n:
        for v in rng.integers(0, V, size=2 * n + 8):
            v = int(v)
            if v not in seen:
                seen.add(v)
                out.append(v)
                if len(out) == n:
                    break
    return np.array(out, np.int32)


def _other_id(rng, V: int, avoid: int) -> int:
    while True:
        v = int(rng.integers(0, V))
        if v != avoid:
            return v


def _plant_unique_max(row: np.ndarray, V: int, idx: int, step: float) -> None:
    """Writes (row max + step) at idx, making idx the only maximal lane."""
    row[idx] = np.float32(row[:V].max() + np.float32(step))


def _store(name, dtype, V, Vp, k_max, vals_f32, gi, drafts, sampled, req, topk, tids, cnts,
           planted, meta=None) -> Workload:
    vals_f32[:, V:] = np.float32(PAD_VALUE)
    logits = bf16_bits(vals_f32) if dtype == "bf16" else vals_f32
    return Workload(name, dtype, V, Vp, k_max, logits, gi.astype(np.int32), drafts.astype(np.int32),
                    sampled.astype(np.int32), req.astype(np.int32), topk.astype(np.int32),
                    tids.astype(np.int32), cnts.astype(np.int32), planted.astype(np.int32),
                    meta or {})


def _verify_drafts(rng, vals, V, gi, p_match, step, drafts, planted, on_bf16_grid=False):
    """For every group, rows j < k get a planted argmax; draft j equals it w.p. p_match."""
    G = gi.shape[0] - 1
    for g in range(G):
        r0, r1 = int(gi[g]), int(gi[g + 1])
        for row in range(r0, r1 - 1):
            idx = int(rng.integers(0, V))
            _plant_unique_max(vals[row], V, idx, step)
            if on_bf16_grid:
                # rounding (max + 1) to BF16 moves it by < 0.25, so it stays the maximum
                vals[row, idx] = bf16_to_f32(bf16_bits(vals[row, idx:idx + 1]))[0]
            planted[row] = idx
            drafts[row] = idx if rng.random() < p_match else _other_id(rng, V, idx)


def tiny(seed: int = SEEDS["tiny"]) -> Workload:
    rng = np.random.default_rng(seed)
    rows, V, Vp = 6, 1000, 1024
    vals = np.zeros((rows, Vp), np.float32)
    vals[:, :V] = np.round(rng.normal(0.0, 2.0, size=(rows, V)) * 8.0) / 8.0
    zero = rng.random((rows, V)) < 0.05
    sign = rng.random((rows, V)) < 0.5
    vals[:, :V][zero & sign] = np.float32(-0.0)
    vals[:, :V][zero & ~sign] = np.float32(0.0)
    gi = np.array([0, 4, 5, 6])
    drafts = np.full(rows, -1, np.int32)
    planted = np.full(rows, -1, np.int32)
    # Row 0: a two-way tie at the maximum (the draft is the smaller id).
    a, b = sorted(_distinct_ids(rng, V, 2).tolist())
    top = np.float32(vals[0, :V].max() + 0.125)
    vals[0, a] = top
    vals[0, b] = top
    planted[0] = a
    drafts[0] = a
    # Row 1: unique planted maximum, matched.  Row 2: planted, not matched.
    for row, match in ((1, True), (2, False)):
        idx = int(rng.integers(0, V))
        _plant_unique_max(vals[row], V, idx, 0.125)
        planted[row] = idx
        drafts[row] = idx if match else _other_id(rng, V, idx)
    G = 3
    req = np.array([1, 1, 0])
    topk = np.array([20, 0, 20])
    tids = np.full((G, MAX_IDS), -1, np.int32)
    extra = _distinct_ids(rng, V, 12, exclude=(3, 7, 999))
    tids[1, :15] = np.concatenate([[7, 999, 3], extra])
    cnts = np.array([0, 15, 0])
    sampled = np.array([-1, int(rng.integers(0, V)), int(rng.integers(0, V))])
    return _store("tiny", "f32", V, Vp, 3, vals, gi, drafts, sampled, req, topk, tids, cnts, planted)


def decode(seed: int = SEEDS["decode"], rows: int = 64) -> Workload:
    rng = np.random.default_rng(seed)
    V, Vp = 151_936, 152_064
    vals = np.empty((rows, Vp), np.float32)
    vals[:, :V] = rng.standard_normal((rows, V), dtype=np.float32) * np.float32(2.5)
    for r in range(rows):
        ids = _distinct_ids(rng, V, 3)
        vals[r, ids] += rng.uniform(12.0, 18.0, size=3).astype(np.float32)
    gi = np.arange(rows + 1)
    drafts = np.full(rows, -1, np.int32)
    sampled = rng.integers(0, V, size=rows)
    req = np.ones(rows)
    topk = np.full(rows, 20)
    tids = np.full((rows, MAX_IDS), -1, np.int32)
    cnts = np.zeros(rows)
    planted = np.full(rows, -1, np.int32)
    return _store("decode", "bf16", V, Vp, 0, vals, gi, drafts, sampled, req, topk, tids, cnts, planted)


def spec(seed: int = SEEDS["spec"], groups: int = 128, V: int = 248_320, Vp: int = 248_448) -> Workload:
    rng = np.random.default_rng(seed)
    k = 3
    rows = groups * (k + 1)
    vals = np.empty((rows, Vp), np.float32)
    vals[:, :V] = rng.standard_normal((rows, V), dtype=np.float32) * np.float32(3.0)
    gi = np.arange(groups + 1) * (k + 1)
    drafts = np.full(rows, -1, np.int32)
    planted = np.full(rows, -1, np.int32)
    _verify_drafts(rng, vals, V, gi, 0.7, 1.0, drafts, planted)
    sampled = np.full(groups, -1)
    req = np.ones(groups)
    ids_mode = (np.arange(groups) % 2) == 0
    topk = np.where(ids_mode, 0, 20)
    tids = np.full((groups, MAX_IDS), -1, np.int32)
    cnts = np.zeros(groups)
    for g in np.nonzero(ids_mode)[0]:
        tids[g] = _distinct_ids(rng, V, MAX_IDS)
        cnts[g] = MAX_IDS
    return _store("spec", "bf16", V, Vp, k, vals, gi, drafts, sampled, req, topk, tids, cnts, planted)


def large(seed: int = SEEDS["large"], groups: int = 256, V: int = 262_144) -> Workload:
    rng = np.random.default_rng(seed)
    k = 7
    rows = groups * (k + 1)
    Vp = V
    vals = np.empty((rows, Vp), np.float32)
    chunk = 64
    for r in range(0, rows, chunk):
        blk = rng.standard_normal((min(chunk, rows - r), V), dtype=np.float32) * np.float32(4.0)
        vals[r:r + blk.shape[0]] = bf16_to_f32(bf16_bits(blk))
    gi = np.arange(groups + 1) * (k + 1)
    drafts = np.full(rows, -1, np.int32)
    planted = np.full(rows, -1, np.int32)
    _verify_drafts(rng, vals, V, gi, 0.6, 1.0, drafts, planted, on_bf16_grid=True)
    sampled = np.full(groups, -1)
    kind = np.arange(groups) % 4          # 0: natural, 1: explicit ids, 2-3: not requested
    req = (kind < 2).astype(np.int32)
    topk = np.where(kind == 0, rng.integers(0, 21, size=groups), 0)
    tids = np.full((groups, MAX_IDS), -1, np.int32)
    cnts = np.zeros(groups)
    for g in np.nonzero(kind == 1)[0]:
        c = int(rng.integers(1, MAX_IDS + 1))
        tids[g, :c] = _distinct_ids(rng, V, c)
        cnts[g] = c
    return _store("large", "f32", V, Vp, k, vals, gi, drafts, sampled, req, topk, tids, cnts, planted)


def wide(seed: int = SEEDS["wide"]) -> Workload:
    rng = np.random.default_rng(seed)
    rows, V, Vp, k = 4, 1_048_576, 1_048_704, 3
    vals = np.empty((rows, Vp), np.float32)
    vals[:, :V] = rng.standard_normal((rows, V), dtype=np.float32)
    bump = rng.random((rows, V)) < 0.01
    vals[:, :V][bump] += np.float32(8.0)
    drafts = np.full(rows, -1, np.int32)
    planted = np.full(rows, -1, np.int32)
    tie_value = np.float32(16.0)           # above N(0,1) + 8 for every lane drawn here
    for r in range(rows):
        ids = _distinct_ids(rng, V, 64)
        vals[r, ids] = tie_value
        planted[r] = int(ids.min())
        if r < k:
            drafts[r] = int(ids.min())
    gi = np.array([0, rows])
    sampled = np.array([-1])
    req = np.array([1])
    topk = np.array([20])
    tids = np.full((1, MAX_IDS), -1, np.int32)
    cnts = np.array([0])
    return _store("wide", "bf16", V, Vp, k, vals, gi, drafts, sampled, req, topk, tids, cnts, planted,
                  meta={"tie_value": float(tie_value)})


def prompt(seed: int = SEEDS["prompt"], rows: int = 512, V: int = 151_936, Vp: int = 152_064,
           dtype: str = "bf16") -> Workload:
    """Prompt scoring: one row per prompt position, N(0,2.5) + 3 spikes of
    +U[12,18]; meta["targets"] holds the scored tokens: a spike id for 30% of
    the rows (a well-predicted token), -1 for 3% (the prompt-end marker), a
    uniform id otherwise."""
    rng = np.random.default_rng(seed)
    vals = np.empty((rows, Vp), np.float32)
    targets = np.empty(rows, np.int32)
    kind = rng.random(rows)
    for r0 in range(0, rows, 64):
        n = min(64, rows - r0)
        vals[r0:r0 + n, :V] = rng.standard_normal((n, V), dtype=np.float32) * np.float32(2.5)
    for r in range(rows):
        ids = _distinct_ids(rng, V, 3)
        vals[r, ids] += rng.uniform(12.0, 18.0, size=3).astype(np.float32)
        targets[r] = ids[int(rng.integers(0, 3))] if kind[r] < 0.3 else (-1 if kind[r] < 0.33
                                                                           else int(rng.integers(0, V)))
    gi = np.arange(rows + 1)
    drafts = np.full(rows, -1, np.int32)
    req = np.ones(rows)
    topk = np.full(rows, 20)
    tids = np.full((rows, MAX_IDS), -1, np.int32)
    cnts = np.zeros(rows)
    planted = np.full(rows, -1, np.int32)
    return _store("prompt", dtype, V, Vp, 0, vals, gi, drafts, targets, req, topk, tids, cnts, planted,
                  meta={"targets": targets})


def commit_clip(w: Workload, seed: int):
    """Per-group commit-clipping inputs (EOS token, output budget) for a block,
    cycling through every case: at the limit (budget 0); EOS on a draft; an EOS
    id drawn at random with a budget of one token; a budget inside the group;
    EOS on a planted row maximum (an accepted draft, or the correction or bonus
    token).  Returns (eos_tokens, budgets), int32 [groups] each."""
    rng = np.random.default_rng(seed)
    gi = np.asarray(w.group_indptr)
    G = w.groups
    eos = np.full(G, -1, np.int32)
    budgets = np.empty(G, np.int32)
    for g in range(G):
        r0, r1 = int(gi[g]), int(gi[g + 1])
        k = r1 - r0 - 1
        kind = g % 5
        budgets[g] = k + 2
        if kind == 0:
            budgets[g] = 0
        elif kind == 1 and k >= 1:
            eos[g] = int(w.draft_tokens[r0 + int(rng.integers(0, k))])
        elif kind == 2:
            eos[g] = int(rng.integers(0, w.V))
            budgets[g] = 1
        elif kind == 3:
            budgets[g] = int(rng.integers(1, k + 2))
        elif kind == 4:
            planted = [int(v) for v in w.planted_argmax[r0:r1] if v >= 0]
            if planted:
                eos[g] = planted[int(rng.integers(0, len(planted)))]
    return eos, budgets


def chain(seed: int = 6, groups: int = 128, k: int = 3, V: int = 248_320, Vp: int = 248_448,
          dtype: str = "bf16", hot: int = 12) -> Workload:
    """Stochastic chain verification inputs: groups of k drafts + 1 bonus row.

    Each row has a small hot set of `hot` seed-drawn ids.  Its logits are N(0,1),
    N(16,1) on the hot set (so that most of the target law's mass is there, as
    when a draft model agrees with the target); its draft law q is a Dirichlet(0.3) draw over the
    hot set (zero elsewhere) mixed with 1% of uniform mass, and the row's draft
    is drawn from q.  Temperatures are U[0.6, 1.4] per group; u (per row) and
    r (per group) are U[0, 1).  Pad lanes hold +1e30 (logits) and 0 (q).
    In meta: draft_probs float32 [rows, Vp], temperature, u, r."""
    rng = np.random.default_rng(seed)
    rows = groups * (k + 1)
    vals = np.full((rows, Vp), np.float32(PAD_VALUE), np.float32)
    vals[:, :V] = rng.standard_normal((rows, V), dtype=np.float32)
    q = np.zeros((rows, Vp), np.float32)
    drafts = np.full(rows, -1, np.int32)
    for r in range(rows):
        ids = rng.choice(V, size=min(hot, V), replace=False)
        vals[r, ids] += np.float32(16.0)
        law = np.full(V, 0.01 / V)
        law[ids] += 0.99 * rng.dirichlet(np.full(ids.size, 0.3))
        law /= law.sum()
        q[r, :V] = law.astype(np.float32)
        if r % (k + 1) != k:
            drafts[r] = int(rng.choice(V, p=law))
    gi = (np.arange(groups + 1) * (k + 1)).astype(np.int32)
    G = groups
    meta = {"draft_probs": q, "temperature": rng.uniform(0.6, 1.4, G).astype(np.float32),
            "u": rng.random(rows, dtype=np.float32), "r": rng.random(G, dtype=np.float32)}
    logits = bf16_bits(vals) if dtype == "bf16" else vals
    return Workload("chain", dtype, V, Vp, k, logits, gi, drafts, np.full(G, -1, np.int32), np.zeros(G, np.int32),
                    np.zeros(G, np.int32), np.full((G, MAX_IDS), -1, np.int32), np.zeros(G, np.int32),
                    np.full(rows, -1, np.int32), meta)


def make(name: str, **kw) -> Workload:
    return {"tiny": tiny, "decode": decode, "spec": spec, "large": large, "wide": wide,
            "prompt": prompt, "chain": chain}[name](**kw)


def custom(rows_f32: np.ndarray, V: int, group_sizes, *, dtype: str = "f32", Vp: int | None = None,
           drafts=None, sampled=None, requested=None, top_k=None, token_ids=None, id_counts=None,
           k_max: int = 15, pad_value: float = PAD_VALUE) -> Workload:
    """Builds a workload from explicit rows (used for hand-made and edge cases).

    ``rows_f32`` holds at least V columns; lanes >= V are replaced by pad_value.
    For dtype="bf16" the values are rounded to BF16.
    """
    rows_f32 = np.asarray(rows_f32, np.float32)
    rows = rows_f32.shape[0]
    if Vp is None:
        Vp = V
    vals = np.full((rows, Vp), np.float32(pad_value), np.float32)
    vals[:, :V] = rows_f32[:, :V]
    sizes = np.asarray(group_sizes, np.int64)
    gi = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    G = sizes.shape[0]
    drafts = np.full(rows, -1, np.int32) if drafts is None else np.asarray(drafts, np.int32)
    sampled = np.full(G, -1, np.int32) if sampled is None else np.asarray(sampled, np.int32)
    requested = np.ones(G, np.int32) if requested is None else np.asarray(requested, np.int32)
    top_k = np.full(G, 20, np.int32) if top_k is None else np.asarray(top_k, np.int32)
    tids = np.full((G, MAX_IDS), -1, np.int32)
    if token_ids is not None:
        for g, lst in enumerate(token_ids):
            if lst is not None and len(lst):
                tids[g, :len(lst)] = lst
    id_counts = np.zeros(G, np.int32) if id_counts is None else np.asarray(id_counts, np.int32)
    planted = np.full(rows, -1, np.int32)
    logits = bf16_bits(vals) if dtype == "bf16" else vals
    return Workload("custom", dtype, V, Vp, k_max, logits, gi, drafts, sampled, requested, top_k,
                    tids, id_counts, planted)
