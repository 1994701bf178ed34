"""Stochastic chain verification on the GPU against the CPU oracle.

The kernel decides acceptance in FP32 from its own lse of x / t, and sums the
draw's FP32 weights in FP64; the oracle works in FP64 throughout.  Where a
decision or a draw is far from its boundary the two must agree exactly; a
decision within a relative 1e-5 of its boundary (u * q(d) against p(d)) may go
either way, and a drawn token must lie in the oracle's inverse-CDF interval
widened by 1e-6 of the total weight.  (FP32 p carries a relative error of a
few 1e-6: ex2 and the rounding of x / t and of lse; the FP64 sums of FP32
weights drift by at most about 3e-7 of the total.)  Those checks recompute p with the
kernel's lse, so that they test the kernel's decisions, not its rounding of
lse, which is compared with the FP64 value separately.
"""
import os

import numpy as np
import pytest

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

DECIDE_REL = 1e-5      # relative band around u * q(d) = p(d)
DRAW_REL = 1e-6        # of the total weight, around r * total
LSE_TOL = 2e-5


def run_gpu_chain(w, plan=None, lse_sentinel=-12345.0):
    import torch
    import logprob_epilogue_gb300 as lpe
    dev = torch.device("cuda", 0)
    if plan is None:
        plan = lpe.Plan(max_rows=max(w.rows, 1), max_groups=max(w.groups, 1), k_max=w.k_max, V=w.V,
                        V_padded=w.Vp, dtype=w.dtype, device=0)
    if w.dtype == "bf16":
        logits = torch.from_numpy(w.logits.view(np.int16)).view(torch.bfloat16).to(dev)
    else:
        logits = torch.from_numpy(w.logits).to(dev)
    ti = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)  # noqa: E731
    tf = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev)  # noqa: E731
    out = dict(accepted=torch.full((max(w.groups, 1),), -7, dtype=torch.int32, device=dev),
               emitted=torch.full((max(w.rows, 1),), -7, dtype=torch.int32, device=dev),
               lse_out=torch.full((max(w.rows, 1),), lse_sentinel, dtype=torch.float32, device=dev),
               status=torch.full((1,), -1, dtype=torch.int32, device=dev))
    m = w.meta
    plan.chain_verify(logits=logits, group_indptr=ti(w.group_indptr), draft_tokens=ti(w.draft_tokens),
                      draft_probs=tf(m["draft_probs"]), temperature=tf(m["temperature"]), u=tf(m["u"]),
                      r=tf(m["r"]), accepted=out["accepted"][:w.groups], emitted=out["emitted"][:w.rows],
                      lse_out=out["lse_out"][:w.rows], status=out["status"])
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy() for k, v in out.items()}
    res["accepted"] = res["accepted"][:w.groups]
    res["emitted"] = res["emitted"][:w.rows]
    res["lse"] = res["lse_out"][:w.rows]
    res["status"] = int(res["status"].view(np.uint32)[0])
    return res, plan


def run_oracle_chain(w):
    m = w.meta
    return oracle.chain_verify(w.logits_f32(), w.V, w.group_indptr, w.draft_tokens, m["draft_probs"],
                               m["temperature"], m["u"], m["r"])


def check_chain(w, gpu, orc):
    """Checks the kernel's outputs.  Returns (groups whose acceptance was
    compared with the oracle's, groups compared with it in full)."""
    x = w.logits_f32()
    q = w.meta["draft_probs"].astype(np.float64)
    temp, u, r = w.meta["temperature"], w.meta["u"], w.meta["r"]
    gi = w.group_indptr
    exact = decided = 0
    assert gpu["status"] == 0, hex(gpu["status"])
    for g in range(w.groups):
        r0, r1 = int(gi[g]), int(gi[g + 1])
        k = r1 - r0 - 1
        t = float(temp[g])
        a = int(gpu["accepted"][g])
        assert 0 <= a <= k, (g, a)
        near = near_decision = False
        for j in range(a + 1):
            row = r0 + j
            xs = x[row, :w.V].astype(np.float64) / t
            lse64 = xs.max() + np.log(np.exp(xs - xs.max()).sum())
            assert abs(float(gpu["lse"][row]) - lse64) <= LSE_TOL * max(1.0, abs(lse64)), (g, j, gpu["lse"][row], lse64)
            lse_k = float(gpu["lse"][row])  # decisions are checked with the kernel's lse
            p = np.exp(xs - lse_k)
            if j < k:
                d = int(w.draft_tokens[row])
                pd = p[d] if 0 <= d < w.V else 0.0
                lhs = float(u[row]) * (q[row, d] if 0 <= d < w.V else 0.0)
                if abs(lhs - pd) <= DECIDE_REL * max(pd, lhs):
                    near = near_decision = True
                elif j < a:
                    assert lhs < pd, (g, j, lhs, pd)
                else:
                    assert lhs >= pd, (g, j, lhs, pd)
            if j < a:
                assert int(gpu["emitted"][row]) == int(w.draft_tokens[row])
                continue
            # the draw at row a
            wts = np.maximum(p - q[row, :w.V], 0.0) if j < k else p
            if wts.sum() <= 0.0:
                wts = p
            cum = np.cumsum(wts)
            tot = cum[-1]
            target = float(r[g]) * tot
            v = int(gpu["emitted"][row])
            assert 0 <= v < w.V and wts[v] > 0.0, (g, v)
            lo = cum[v] - wts[v]
            band = DRAW_REL * tot
            assert lo <= target + band and target - band < cum[v], (g, v, lo, target, cum[v])
            if abs(target - lo) <= band or abs(target - cum[v]) <= band:
                near = True
        assert (gpu["emitted"][r0 + a + 1:r1] == -1).all()
        assert (gpu["lse"][r0 + a + 1:r1] == np.float32(-12345.0)).all()  # rows past the prefix are not read
        if not near_decision:
            decided += 1
            assert int(orc["accepted"][g]) == a, (g, orc["accepted"][g], a)
        if not near:
            exact += 1
            assert (orc["emitted_tokens"][r0:r1] == gpu["emitted"][r0:r1]).all(), g
    return decided, exact


@pytest.mark.parametrize("dtype,V,Vp", [("bf16", 20_000, 20_000), ("bf16", 40_001, 40_008), ("f32", 33_333, 33_336),
                                         ("f32", 8_191, 8_192)])
@pytest.mark.parametrize("k", [1, 3, 7])
def test_chain_matches_oracle(dtype, V, Vp, k):
    w = W.chain(seed=100 + k + V % 97, groups=40, k=k, V=V, Vp=Vp, dtype=dtype)
    gpu, plan = run_gpu_chain(w)
    decided, exact = check_chain(w, gpu, run_oracle_chain(w))
    plan.close()
    assert decided >= w.groups - 2 and exact >= w.groups // 4, (decided, exact)
    # the workload exercises acceptances, rejections and full acceptances
    acc = gpu["accepted"]
    assert (acc == 0).any() and (acc > 0).any()


def test_chain_full_size():
    w = W.chain()  # 128 groups x (3 + 1) rows x 248,320 BF16
    gpu, plan = run_gpu_chain(w)
    decided, exact = check_chain(w, gpu, run_oracle_chain(w))
    plan.close()
    assert decided >= w.groups - 2 and exact >= w.groups // 4, (decided, exact)


def test_chain_preserves_the_target_law():
    # The defining property, through the kernel: every draft id d weighted by
    # q(d), u and r on midpoint grids of N points; the first emitted token must
    # follow p, the bonus token after an acceptance the bonus row's law, and
    # the acceptance rate must be sum_d min(q(d), p(d)), each within ~1/N.
    V, Vp, N, t = 5, 8, 160, 0.7
    rng = np.random.default_rng(81)
    x0 = rng.normal(0.0, 1.5, V).astype(np.float32)
    x1 = rng.normal(0.0, 1.5, V).astype(np.float32)
    q = rng.dirichlet(np.ones(V)).astype(np.float32)
    grid = (np.arange(N) + 0.5) / N
    d, ui, ri = np.meshgrid(np.arange(V), np.arange(N), np.arange(N), indexing="ij")
    d, ui, ri = d.ravel(), ui.ravel(), ri.ravel()
    G = d.size
    rows = np.full((2 * G, Vp), 1e30, np.float32)
    rows[0::2, :V], rows[1::2, :V] = x0, x1
    qq = np.zeros((2 * G, Vp), np.float32)
    qq[0::2, :V] = q
    drafts = np.full(2 * G, -1, np.int32)
    drafts[0::2] = d
    u = np.zeros(2 * G, np.float32)
    u[0::2] = grid[ui]
    w = W.custom(rows, V, [2] * G, Vp=Vp, drafts=drafts, k_max=1)
    w.meta = {"draft_probs": qq, "temperature": np.full(G, t, np.float32), "u": u,
              "r": grid[ri].astype(np.float32)}
    gpu, plan = run_gpu_chain(w)
    plan.close()
    assert gpu["status"] == 0
    law = lambda x: np.exp(x / t - np.log(np.exp(x.astype(np.float64) / t).sum()))  # noqa: E731
    wgt = q[d].astype(np.float64) / (N * N)
    freq = np.bincount(gpu["emitted"][0::2], weights=wgt, minlength=V)
    assert np.abs(freq - law(x0)).max() < 3.0 / N, (freq, law(x0))
    acc = gpu["accepted"] == 1
    bonus = np.bincount(gpu["emitted"][1::2][acc], weights=wgt[acc], minlength=V) / wgt[acc].sum()
    assert np.abs(bonus - law(x1)).max() < 3.0 / N, (bonus, law(x1))
    rate = float(np.minimum(q.astype(np.float64), law(x0)).sum())
    assert abs(float(wgt[acc].sum()) - rate) < 2.0 / N
    # and the kernel agrees with the oracle on the same grid, away from boundaries
    orc = run_oracle_chain(w)
    agree = (orc["accepted"] == gpu["accepted"]).mean()
    assert agree > 0.99, agree


def test_chain_bad_inputs_and_bonus_only_groups():
    V, Vp = 1000, 1000
    rng = np.random.default_rng(7)
    x = rng.normal(0, 2, (7, V)).astype(np.float32)
    q = np.zeros((7, Vp), np.float32)
    q[:, :V] = rng.dirichlet(np.ones(V), 7).astype(np.float32)
    # groups: [0,1] k=1 with a draft >= V; [2] k=0 (bonus only); [3,4] bad temperature; [5,6] k=1 valid
    drafts = np.array([V + 5, -1, -1, 3, -1, 10, -1], np.int32)
    w = W.custom(x, V, [2, 1, 2, 2], Vp=Vp, drafts=drafts, k_max=3)
    w.meta = {"draft_probs": q, "temperature": np.array([1.0, 0.8, 0.0, 1.2], np.float32),
              "u": rng.random(7, dtype=np.float32), "r": rng.random(4, dtype=np.float32)}
    gpu, plan = run_gpu_chain(w)
    plan.close()
    assert gpu["status"] == 0x2 | 0x20, hex(gpu["status"])
    assert gpu["accepted"][0] == 0 and gpu["accepted"][1] == 0 and gpu["accepted"][2] == -1
    assert gpu["emitted"][3] == -1 and gpu["emitted"][4] == -1
    # the valid groups still match the checks (bad ones removed)
    keep = [0, 1, 3]
    sub = W.custom(x[[0, 1, 2, 5, 6]], V, [2, 1, 2], Vp=Vp, drafts=drafts[[0, 1, 2, 5, 6]], k_max=3)
    sub.meta = {"draft_probs": q[[0, 1, 2, 5, 6]], "temperature": w.meta["temperature"][keep],
                "u": w.meta["u"][[0, 1, 2, 5, 6]], "r": w.meta["r"][keep]}
    gsub = {"accepted": gpu["accepted"][keep], "emitted": gpu["emitted"][[0, 1, 2, 5, 6]],
            "lse": gpu["lse"][[0, 1, 2, 5, 6]], "status": 0}
    check_chain(sub, gsub, run_oracle_chain(sub))
