"""Draws placed at inverse-CDF boundaries: the precise redraw.

For each sequence the draw uniform of its final (correction or bonus) draw is
replaced by the float32 value nearest above, or nearest below, a CDF boundary
of the oracle's draw distribution: u lands within one float32 spacing (about
3e-8) of the boundary, where single-precision running sums cannot decide the
token.  The library must flag such draws and redraw them precisely, so the
GPU token must equal the oracle's in every case whose oracle margin exceeds
1e-12 (the double-float redraw's error is below 1e-11 of the mass; closer
cases are counted as excused).
"""

import numpy as np
import pytest
import torch

from gpu_helpers import oracle_chain, oracle_tree, run_chain, run_tree
from oracle import philox
from oracle.policy import policy_distribution
from speculative_decoding_verification_temp_gb300 import workloads

pytestmark = pytest.mark.gpu

# "stream": the streaming paths (the chain path, the tree walk); "resident": an
# all-off top-k array selects the resident cluster kernel on the same inputs
PATHS = ["stream", "resident"]
TIE = 1e-12


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()


def philox_override(seed, nseq, npos):
    u = np.zeros((nseq, npos, 2), np.float32)
    for s in range(nseq):
        for i in range(npos):
            for d in range(2):
                u[s, i, d] = philox.uniform(seed, s, i, d)
    return u


def near_boundary(weights, rng, above):
    """A float32 u within one spacing of a CDF boundary of `weights`."""
    c = np.cumsum(np.asarray(weights, np.float64))
    total = c[-1]
    cand = np.flatnonzero((weights > 1e-4 * total) & (np.concatenate([[0.0], c[:-1]]) > 0.05 * total)
                          & (np.concatenate([[0.0], c[:-1]]) < 0.95 * total))
    if cand.size == 0:
        return None
    v = int(rng.choice(cand))
    b = c[v - 1] / total
    u = np.float32(b)
    if above and float(u) <= b:
        u = np.nextafter(u, np.float32(1))
    if not above and float(u) >= b:
        u = np.nextafter(u, np.float32(0))
    return u


def chain_draw_weights(w, r):
    """The distribution a chain's final token is drawn from (oracle)."""
    if r["final_dist"] is not None:
        return r["final_dist"]
    b, j = r["seq"], r["num_accepted"]
    d = policy_distribution(w["target"][b, j], w["target_temperature"][b], w["target_top_k"][b])
    return None if d.onehot else d.probs


def tree_draw_weights(w, r):
    if r["final_dist"] is not None:
        return r["final_dist"]
    t = r["tree"]
    node = r["path"][r["num_accepted"]]
    d = policy_distribution(w["target"][t, node], w["target_temperature"][t],
                            w["target_top_k"][t])
    return None if d.onehot else d.probs


def check(gpu_tokens, gpu_num, want, key, log, label):
    checked = 0
    for r in want:
        s = r[key]
        same = gpu_num[s] == r["num_accepted"] and list(gpu_tokens[s]) == list(r["tokens"])
        if same:
            checked += 1
            continue
        assert r["draw_margin"] is not None and r["draw_margin"] <= TIE, (
            f"{label} {key} {s}: gpu {gpu_num[s]} {list(gpu_tokens[s])} "
            f"oracle {r['num_accepted']} {r['tokens']} margin {r['draw_margin']}")
        log.excuse(f"{label} {key} {s}", r["draw_margin"])
    return checked


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_chain_draws_at_boundaries(dtype, path, exception_log):
    w = workloads.make_chain(48, 3, 128256 if dtype == "bf16" else 65536, dtype=dtype, seed=31,
                             sigma=0.6)
    uo = philox_override(w["seed"], 48, 4)
    rng = np.random.default_rng(5)
    for r in oracle_chain(w, uniform_override=uo):
        wt = chain_draw_weights(w, r)
        if wt is None:
            continue
        u = near_boundary(wt, rng, above=r["seq"] % 2 == 0)
        if u is not None:
            uo[r["seq"], r["num_accepted"], 1] = u
    want = oracle_chain(w, uniform_override=uo)
    exception_log.add_rows(len(want) * 4)
    res = run_chain(w, uniform_override=uo, force_resident=path == "resident")
    n = check(res.tokens.cpu().numpy(), res.num_accepted.cpu().numpy(), want, "seq",
              exception_log, f"boundary-chain-{dtype}-{path}")
    assert n >= 40


@pytest.mark.parametrize("path", PATHS)
def test_tree_draws_at_boundaries(path, exception_log):
    # sigma 0.9: many rejected siblings, so held residuals after several
    # rejections (c_s with s > 1) are redrawn too
    w = workloads.make_tree(16, 30, 128256, dtype="bf16", seed=32, sigma=0.9,
                            branching=(4, 3, 2))
    uo = philox_override(w["seed"], 16, 30)
    rng = np.random.default_rng(6)
    for r in oracle_tree(w, uniform_override=uo):
        if r["num_accepted"] < 0:
            continue
        wt = tree_draw_weights(w, r)
        if wt is None:
            continue
        u = near_boundary(wt, rng, above=r["tree"] % 2 == 1)
        if u is not None:
            uo[r["tree"], r["path"][r["num_accepted"]], 1] = u
    want = oracle_tree(w, uniform_override=uo)
    exception_log.add_rows(len(want) * 30)
    res = run_tree(w, uniform_override=uo, force_resident=path == "resident")
    toks = res.tokens.cpu().numpy()
    n = check(toks, res.num_accepted.cpu().numpy(), want, "tree", exception_log,
              f"boundary-tree-{path}")
    assert n >= 12


@pytest.mark.parametrize("path", PATHS)
def test_chain_draws_at_boundaries_with_equal_entries(path, exception_log):
    """Draft rows that are the target rows with a few entries swapped: S_p =
    S_q, so p = q on every other entry and [p - q]_+ lives on the swapped
    entries alone.  Every entry with p = q sits on the edge of the residual's
    support, which the precise redraw must treat exactly (its fast
    classification of entries cannot decide them)."""
    B, gamma, V = 12, 2, 4096
    rng = np.random.default_rng(11)
    target = workloads.round_bf16_inplace(
        (2.0 * rng.standard_normal((B, gamma + 1, V))).astype(np.float32))
    draft = target[:, :gamma].copy()
    tokens = np.zeros((B, gamma), np.int32)
    for b in range(B):
        for i in range(gamma):
            row = draft[b, i]
            order = np.argsort(row)
            # swap eight pairs of entries far apart in value (p and q differ there)
            lo, hi = order[:8], order[-8:]
            row[lo], row[hi] = target[b, i, hi], target[b, i, lo]
            tokens[b, i] = lo[0]  # now q(x) > p(x): a likely rejection
    w = dict(kind="chain", B=B, gamma=gamma, V=V, dtype="bf16", target=target, draft=draft,
             tokens=tokens, target_temperature=np.ones(B, np.float32),
             draft_temperature=np.ones(B, np.float32), target_top_k=None, draft_top_k=None,
             seed=77)
    uo = philox_override(w["seed"], B, gamma + 1)
    uo[:, :, 0] = np.float32(0.99999)  # reject at the first position
    prng = np.random.default_rng(12)
    for r in oracle_chain(w, uniform_override=uo):
        wt = chain_draw_weights(w, r)
        if wt is None:
            continue
        u = near_boundary(wt, prng, above=r["seq"] % 2 == 0)
        if u is not None:
            uo[r["seq"], r["num_accepted"], 1] = u
    want = oracle_chain(w, uniform_override=uo)
    assert sum(r["num_accepted"] < gamma for r in want) >= B // 2
    exception_log.add_rows(len(want) * (gamma + 1))
    res = run_chain(w, uniform_override=uo, force_resident=path == "resident")
    n = check(res.tokens.cpu().numpy(), res.num_accepted.cpu().numpy(), want, "seq",
              exception_log, f"boundary-equal-entries-{path}")
    assert n >= B - 2
