"""Helpers of the GPU parity tests: run the CUDA path and the oracle on the
same seeded inputs and compare them under the verification's rules.

Integer outputs must match exactly.  A disagreement is excused only when the
oracle shows it sits within rounding of a decision: |u - alpha| <= 1e-5 at the
first differing acceptance test, or an inverse-CDF boundary within 1e-5 of the
draw uniform; excused rows are logged and counted against the 1e-5 budget.
Residual probabilities must match within 1e-5 (fp32 logits) or 2e-3 (bf16).
"""

import numpy as np
import torch

import speculative_decoding_verification_temp_gb300 as sv
from oracle import verify as ov

MARGIN = 1e-5
RESID_TOL = {"f32": 1e-5, "bf16": 2e-3}


def top_k_arg(k, V, force_resident):
    """The top-k argument of a call: None when no row filters (every k <= 0 or
    >= V), the array itself otherwise.  force_resident passes it as a CUDA
    tensor even when every row is off: the binding forwards a device array as
    given, and for trees any top-k array selects the resident kernel (chains
    take the chain path with or without one; run_chain forces the resident
    kernel with unaligned rows instead)."""
    if k is None:
        return None
    k = np.asarray(k)
    if force_resident:
        return torch.from_numpy(np.ascontiguousarray(k, dtype=np.int32)).cuda()
    if np.any((k > 0) & (k < V)):
        return k
    return None


def to_dev(arr, dtype):
    t = torch.from_numpy(np.ascontiguousarray(arr)).cuda()
    return t.to(torch.bfloat16) if dtype == "bf16" else t


def run_chain(w, uniform_override=None, return_residual=False, seed=None, pad_to=None,
              workspace_tensor=None, force_resident=False):
    """Chain verification of workload w through the binding.  force_resident:
    rows one entry longer than V (not 16-byte aligned), which only the
    resident kernel takes."""
    dt = w["dtype"]
    target = w["target"]
    if force_resident and pad_to is None:
        pad_to = target.shape[-1] + 1
    draft = w["draft"]
    if pad_to is not None:
        V = target.shape[-1]
        tp = np.zeros(target.shape[:-1] + (pad_to,), np.float32)
        tp[..., :V] = target
        dp = np.zeros(draft.shape[:-1] + (pad_to,), np.float32)
        dp[..., :V] = draft
        t_dev = to_dev(tp, dt)[..., :V]
        d_dev = to_dev(dp, dt)[..., :V]
    else:
        t_dev, d_dev = to_dev(target, dt), to_dev(draft, dt)
    res = sv.verify_chain(
        t_dev, d_dev, torch.from_numpy(w["tokens"]).cuda(),
        w["target_temperature"], w["draft_temperature"],
        target_top_k=top_k_arg(w.get("target_top_k"), w["target"].shape[-1], force_resident),
        draft_top_k=top_k_arg(w.get("draft_top_k"), w["target"].shape[-1], force_resident),
        seed=w["seed"] if seed is None else seed,
        uniform_override=None if uniform_override is None else torch.from_numpy(
            np.ascontiguousarray(uniform_override, dtype=np.float32)).cuda(),
        return_residual=return_residual, workspace_tensor=workspace_tensor)
    torch.cuda.synchronize()
    return res


def oracle_chain(w, uniform_override=None, seed=None, seqs=None):
    return ov.verify_chain(w["target"], w["draft"], w["tokens"], w["target_temperature"],
                           w["draft_temperature"], w.get("target_top_k"), w.get("draft_top_k"),
                           seed=w["seed"] if seed is None else seed,
                           uniform_override=uniform_override, seqs=seqs)


def compare_chain(res, want, log, label, dtype="bf16", check_residual=False):
    """Compare GPU chain results with oracle results (list of per-seq dicts)."""
    n = res.num_accepted.cpu().numpy()
    toks = res.tokens.cpu().numpy()
    flags = res.flags.cpu().numpy().astype(np.int64) & 0xFFFFFFFF
    resid = res.residual.cpu().numpy() if check_residual else None
    gamma = toks.shape[1] - 1
    log.add_rows(len(want) * (gamma + 1))
    failures = []
    for r in want:
        b = r["seq"]
        same = (n[b] == r["num_accepted"] and list(toks[b]) == r["tokens"]
                and flags[b] == r["flags"])
        if same:
            if check_residual:
                fd = r["final_dist"]
                ref = np.zeros(resid.shape[1]) if fd is None else np.asarray(fd, np.float64)
                err = np.abs(resid[b] - ref).max()
                if err > RESID_TOL[dtype]:
                    failures.append(f"{label} seq {b}: residual error {err:.3e}")
            continue
        margin = excuse_margin_chain(n[b], toks[b], r)
        if margin is not None and margin <= MARGIN and flags[b] == r["flags"]:
            log.excuse(f"{label} seq {b}", margin)
            continue
        failures.append(f"{label} seq {b}: gpu j={n[b]} toks={list(toks[b])} flags={flags[b]} | "
                        f"oracle j={r['num_accepted']} toks={r['tokens']} flags={r['flags']} "
                        f"margin={margin}")
    assert not failures, "\n".join(failures[:20])


def excuse_margin_chain(j_gpu, toks_gpu, r):
    """Oracle margin at the first point where the GPU result departs from it."""
    j = r["num_accepted"]
    if j_gpu != j:
        pos = min(j_gpu, j)
        for i, m in r["decisions"]:
            if i == pos:
                return m
        return None
    if r["draw_margin"] is None:
        return None
    return r["draw_margin"]


def run_tree(w, uniform_override=None, return_residual=False, seed=None, workspace_tensor=None,
             force_resident=False):
    dt = w["dtype"]
    res = sv.verify_tree(
        to_dev(w["target"], dt), to_dev(w["draft"], dt), torch.from_numpy(w["tokens"]).cuda(),
        torch.from_numpy(w["parent"]).cuda(), w["max_depth"], w["target_temperature"],
        w["draft_temperature"],
        target_top_k=top_k_arg(w.get("target_top_k"), w["target"].shape[-1], force_resident),
        draft_top_k=top_k_arg(w.get("draft_top_k"), w["target"].shape[-1], force_resident),
        seed=w["seed"] if seed is None else seed,
        uniform_override=None if uniform_override is None else torch.from_numpy(
            np.ascontiguousarray(uniform_override, dtype=np.float32)).cuda(),
        return_residual=return_residual, workspace_tensor=workspace_tensor)
    torch.cuda.synchronize()
    return res


def oracle_tree(w, uniform_override=None, seed=None, trees=None):
    want = ov.verify_tree(w["target"], w["draft"], w["tokens"], w["parent"], w["max_depth"],
                          w["target_temperature"], w["draft_temperature"],
                          w.get("target_top_k"), w.get("draft_top_k"),
                          seed=w["seed"] if seed is None else seed,
                          uniform_override=uniform_override, trees=trees)
    for r in want:
        r["rows"] = w["parent"].shape[1]  # a tree is N target rows
    return want


def compare_tree(res, want, log, label, dtype="bf16", check_residual=False):
    n = res.num_accepted.cpu().numpy()
    path = res.path.cpu().numpy()
    toks = res.tokens.cpu().numpy()
    flags = res.flags.cpu().numpy().astype(np.int64) & 0xFFFFFFFF
    resid = res.residual.cpu().numpy() if check_residual else None
    failures = []
    for r in want:
        t = r["tree"]
        log.add_rows(r.get("rows", 1))
        same = (n[t] == r["num_accepted"] and list(path[t]) == r["path"]
                and list(toks[t]) == r["tokens"] and flags[t] == r["flags"])
        if same:
            if check_residual:
                fd = r["final_dist"]
                ref = np.zeros(resid.shape[1]) if fd is None else np.asarray(fd, np.float64)
                err = np.abs(resid[t] - ref).max()
                if err > RESID_TOL[dtype]:
                    failures.append(f"{label} tree {t}: residual error {err:.3e}")
            continue
        margins = [m for _, m in r["decisions"]]
        if r["draw_margin"] is not None:
            margins.append(r["draw_margin"])
        margin = min(margins) if margins else None
        if margin is not None and margin <= MARGIN:
            log.excuse(f"{label} tree {t}", margin)
            continue
        failures.append(f"{label} tree {t}: gpu n={n[t]} path={list(path[t])} toks={list(toks[t])} "
                        f"flags={flags[t]} | oracle n={r['num_accepted']} path={r['path']} "
                        f"toks={r['tokens']} flags={r['flags']}")
    assert not failures, "\n".join(failures[:20])
