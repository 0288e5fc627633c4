"""Top-p and min-p on the GPU against the oracle.

wineandchord.com "推测解码：接受规则、状态与收益边界", § 与 Logit Processor 的组合
lists top-p and min-p among the processors that p and q must both reflect;
the oracle applies the published definitions (oracle.policy:
temperature and top-k, then top-p, then min-p, each renormalised, ties at a
boundary kept).

Integer outputs must match the oracle exactly.  A sequence may differ only
where the oracle shows a decision within rounding: |u - alpha| <= 1e-5, a draw
within 1e-5 of a CDF boundary, or a filter boundary within 1e-5 (top_p within
1e-5 of a cumulative mass of the sorted distribution, or min_p within 1e-5
relative of a probability ratio p(x) / max p).  Such sequences are logged
with the session's exception log and count against its 1e-5-of-rows budget.
Residuals are compared within the dtype's tolerance wherever the integers
agree.
"""

import numpy as np
import pytest
import torch

from gpu_helpers import MARGIN, RESID_TOL, excuse_margin_chain, to_dev
from oracle import policy as pol
from oracle import verify as ov
from speculative_decoding_verification_temp_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()


def filter_margin(z, T, top_k, top_p, min_p):
    """Smallest oracle-side distance of a row's filter parameters from a
    boundary: top_p from any cumulative mass of the sorted distribution after
    temperature and top-k, min_p (relative) from any ratio p(x) / max p after
    top-p.  inf when the row is greedy, not finite or unfiltered."""
    d = pol.policy_distribution(z, T, top_k)
    if d.onehot:
        return np.inf
    m = np.inf
    probs = d.probs
    tp = float(top_p)
    if tp < 1.0:
        cum = np.cumsum(np.sort(probs)[::-1])
        m = min(m, float(np.abs(cum - tp).min()))
        probs = pol.topp_filter(probs, tp)
    mp = float(min_p)
    if mp > 0.0:
        mp = min(mp, 1.0)
        kept = probs[probs > 0]
        ratio = kept / kept.max()
        m = min(m, float((np.abs(ratio - mp) / mp).min()))
    return m


def run_and_compare(w, P, M, log, label, PQ=None, MQ=None, check_residual=True):
    """Verify chain workload w with per-sequence top-p P and min-p M on the
    target side (PQ / MQ on the draft side, default the same) and compare with
    the oracle."""
    import speculative_decoding_verification_temp_gb300 as sv
    dt = w["dtype"]
    PQ = P if PQ is None else PQ
    MQ = M if MQ is None else MQ
    kp, kq = w.get("target_top_k"), w.get("draft_top_k")
    kp_arg = None if kp is None or not np.any((kp > 0) & (kp < w["V"])) else kp
    kq_arg = None if kq is None or not np.any((kq > 0) & (kq < w["V"])) else kq
    r = sv.verify_chain(to_dev(w["target"], dt), to_dev(w["draft"], dt),
                        torch.from_numpy(w["tokens"]).cuda(), w["target_temperature"],
                        w["draft_temperature"], target_top_k=kp_arg, draft_top_k=kq_arg,
                        seed=w["seed"], target_top_p=P, draft_top_p=PQ, target_min_p=M,
                        draft_min_p=MQ, return_residual=check_residual)
    torch.cuda.synchronize()
    want = ov.verify_chain(w["target"], w["draft"], w["tokens"], w["target_temperature"],
                           w["draft_temperature"], kp, kq, seed=w["seed"], target_top_p=P,
                           draft_top_p=PQ, target_min_p=M, draft_min_p=MQ)
    n, toks = r.num_accepted.cpu().numpy(), r.tokens.cpu().numpy()
    flags = r.flags.cpu().numpy().astype(np.int64) & 0xFFFFFFFF
    resid = r.residual.cpu().numpy() if check_residual else None
    gamma = toks.shape[1] - 1
    log.add_rows(len(want) * (gamma + 1))
    failures = []
    for x in want:
        b = x["seq"]
        if n[b] == x["num_accepted"] and list(toks[b]) == x["tokens"] and flags[b] == x["flags"]:
            if check_residual:
                fd = x["final_dist"]
                ref = np.zeros(resid.shape[1]) if fd is None else np.asarray(fd, np.float64)
                err = np.abs(resid[b] - ref).max()
                if err > RESID_TOL[dt]:
                    failures.append(f"{label} seq {b}: residual error {err:.3e}")
            continue
        margins = []
        m0 = excuse_margin_chain(n[b], toks[b], x)
        if m0 is not None:
            margins.append(m0)
        zt = np.asarray(w["target"][b], np.float64)
        zd = np.asarray(w["draft"][b], np.float64)
        kpb = 0 if kp is None else int(kp[b])
        kqb = 0 if kq is None else int(kq[b])
        for i in range(gamma + 1):
            margins.append(filter_margin(zt[i], w["target_temperature"][b], kpb, P[b], M[b]))
        for i in range(gamma):
            margins.append(filter_margin(zd[i], w["draft_temperature"][b], kqb, PQ[b], MQ[b]))
        margin = min(margins) if margins else np.inf
        if margin <= MARGIN and flags[b] == x["flags"]:
            log.excuse(f"{label} seq {b}", margin)
            continue
        failures.append(f"{label} seq {b}: gpu j={n[b]} toks={list(toks[b])} flags={flags[b]} | "
                        f"oracle j={x['num_accepted']} toks={x['tokens']} flags={x['flags']} "
                        f"margin={margin}")
    assert not failures, "\n".join(failures[:20])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("tp,mp", [(0.9, 0.0), (1.0, 0.05), (0.9, 0.05), (0.5, 0.02),
                                   (0.0, 0.0)])
def test_chain_top_p_min_p(dtype, tp, mp, exception_log):
    # ragged V (not a multiple of 8), both sides filtered alike
    w = workloads.make_chain(16, 4, 4099, dtype=dtype, seed=91)
    B = w["B"]
    run_and_compare(w, np.full(B, tp, np.float32), np.full(B, mp, np.float32), exception_log,
                    f"{dtype} top_p={tp} min_p={mp}")


def test_chain_filters_full_vocabulary(exception_log):
    # the c2 recipe (V = 128256 bf16, temperature 1, draft sigma 0.4) with
    # top-p 0.9 and min-p 0.05 on both sides
    c = dict(workloads.CONFIGS[2])
    c.pop("kind")
    c["B"] = 12
    w = workloads.make_chain(seed=1002, **c)
    B = w["B"]
    run_and_compare(w, np.full(B, 0.9, np.float32), np.full(B, 0.05, np.float32),
                    exception_log, "c2 shape top_p=0.9 min_p=0.05")


def test_chain_filters_mixed_per_sequence(exception_log):
    # per-sequence parameters, some rows unfiltered, with top-k, greedy rows
    # and different draft-side filters
    w = workloads.make_chain(24, 5, 20000, dtype="bf16", seed=93, greedy_seqs=4, top_k=40)
    rng = np.random.default_rng(5)
    B = w["B"]
    P = rng.choice(np.array([1.0, 0.95, 0.8, 0.3], np.float32), B)
    M = rng.choice(np.array([0.0, 0.01, 0.1], np.float32), B)
    PQ = rng.choice(np.array([1.0, 0.9], np.float32), B)
    MQ = rng.choice(np.array([0.0, 0.05], np.float32), B)
    run_and_compare(w, P, M, exception_log, "mixed filters", PQ=PQ, MQ=MQ)


def test_chain_filters_with_boundary_ties(exception_log):
    # logits from a handful of values: every filter boundary falls inside a
    # large group of tied entries, which are all kept
    w = workloads.make_chain(16, 3, 3001, dtype="bf16", seed=95)
    rng = np.random.default_rng(6)
    levels = np.array([2.0, 1.0, 0.0, -1.0, -3.0], np.float32)
    w["target"] = rng.choice(levels, w["target"].shape).astype(np.float32)
    gamma = w["draft"].shape[1]
    w["draft"] = np.clip(w["target"][:, :gamma] + rng.choice(np.array([0.0, 1.0, -1.0], np.float32),
                                                             w["draft"].shape), -3, 2).astype(np.float32)
    B = w["B"]
    run_and_compare(w, np.full(B, 0.6, np.float32), np.full(B, 0.3, np.float32), exception_log,
                    "tied logits")


def test_chain_filter_out_of_range_readings(exception_log):
    # NaN switches a filter off, top_p <= 0 keeps the most probable value,
    # min_p > 1 is taken as 1
    w = workloads.make_chain(12, 3, 5003, dtype="f32", seed=97)
    B = w["B"]
    P = np.array([np.nan, -2.0, 0.0, 1.5] * 3, np.float32)
    M = np.array([3.0, np.nan, -1.0, 1.0] * 3, np.float32)
    run_and_compare(w, P, M, exception_log, "out-of-range filters")


def test_tree_filters(exception_log):
    import speculative_decoding_verification_temp_gb300 as sv
    from gpu_helpers import compare_tree
    w = workloads.make_tree(6, 20, 4096, dtype="bf16", seed=99, branching=(3, 2, 2))
    T = w["parent"].shape[0]
    P = np.full(T, 0.85, np.float32)
    M = np.full(T, 0.02, np.float32)
    r = sv.verify_tree(to_dev(w["target"], "bf16"), to_dev(w["draft"], "bf16"),
                       torch.from_numpy(w["tokens"]).cuda(), torch.from_numpy(w["parent"]).cuda(),
                       w["max_depth"], w["target_temperature"], w["draft_temperature"],
                       seed=w["seed"], target_top_p=P, draft_top_p=P, target_min_p=M,
                       draft_min_p=M, return_residual=True)
    torch.cuda.synchronize()
    want = ov.verify_tree(w["target"], w["draft"], w["tokens"], w["parent"], w["max_depth"],
                          w["target_temperature"], w["draft_temperature"], seed=w["seed"],
                          target_top_p=P, draft_top_p=P, target_min_p=M, draft_min_p=M)
    for x in want:
        x["rows"] = w["parent"].shape[1]
    compare_tree(r, want, exception_log, "tree filters", dtype="bf16", check_residual=True)
