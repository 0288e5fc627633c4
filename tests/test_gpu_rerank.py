"""EAGLE-2 rerank on the GPU against the oracle.

The oracle ranks the exact path products (zzszmyf.github.io "LLM
推测解码精读笔记 · 04 EAGLE", § 10.3 扩展 + 重排); the kernel ranks float32
products, each product rounded once per level.  Counts and flags must match
exactly.  The kept set must match exactly too, except where the exact values
at the cut lie within the float32 rounding bound of each other (or both below
the float32 normal range), where either choice is correct up to rounding:
such trees are logged with the session's exception log.  Every kept value must
be within that rounding bound of its exact product.
"""

import numpy as np
import pytest
import torch

from oracle import verify as ov
from speculative_decoding_verification_temp_gb300 import workloads

pytestmark = pytest.mark.gpu

ULP = 2.0 ** -24        # unit roundoff of float32
TINY = 2.0 ** -125      # below this a float32 product may be flushed or subnormal


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()


def close_values(a, da, b, db):
    """Exact values a (depth da) and b (depth db) that float32 products taken
    level by level may not order correctly."""
    if a < TINY and b < TINY:
        return True
    return abs(a - b) <= (da + db + 2) * ULP * max(a, b)


def run_and_check(parent, conf, m, log):
    import speculative_decoding_verification_temp_gb300 as sv
    r = sv.tree_rerank(torch.from_numpy(parent).cuda(), torch.from_numpy(conf).cuda(), m)
    torch.cuda.synchronize()
    nodes, newp, val = r.nodes.cpu().numpy(), r.parent.cpu().numpy(), r.value.cpu().numpy()
    count, flags = r.count.cpu().numpy(), r.flags.cpu().numpy()
    log.add_rows(parent.shape[0])
    for t in range(parent.shape[0]):
        wn, wp, wv, wf = ov.tree_rerank(parent[t], conf[t], m)
        k = len(wn)
        assert count[t] == k and flags[t] == wf, (t, count[t], k, flags[t], wf)
        assert (nodes[t, k:] == -1).all() and (newp[t, k:] == -1).all()
        if k == 0:
            continue
        got = [int(x) for x in nodes[t, :k]]
        order, value, depth = ov.rerank_order(parent[t], conf[t])
        exact = [ov.value_float(v) for v in value]
        if got != wn:
            # only nodes whose exact values sit within rounding of the cut
            cut = order[k - 1]
            diff = set(got) ^ set(wn)
            assert all(close_values(exact[n], depth[n], exact[cut], depth[cut]) for n in diff), \
                (t, sorted(diff), exact[cut])
            log.excuse(f"rerank tree {t} m={m}: kept sets differ at {sorted(diff)}",
                       max(abs(exact[n] - exact[cut]) / max(exact[cut], TINY) for n in diff))
        # the kernel's kept set is connected and re-indexed consistently
        pos = {n: i for i, n in enumerate(got)}
        assert got == sorted(got) and got[0] == 0
        assert list(newp[t, :k]) == [-1 if n == 0 else pos[int(parent[t, n])] for n in got]
        for i, n in enumerate(got):
            tol = (depth[n] + 1) * ULP * exact[n] + TINY
            assert abs(float(val[t, i]) - exact[n]) <= tol, (t, n, float(val[t, i]), exact[n])
    return r


@pytest.mark.parametrize("N", [1, 2, 17, 60, 1000, 4096])
def test_rerank_random_trees(N, exception_log):
    w = workloads.make_rerank(6, N, seed=70 + N)
    for m in sorted({1, 5, 64, N, N + 3}):
        run_and_check(w["parent"], w["confidence"], m, exception_log)


def test_rerank_deep_chain_and_coarse_ties(exception_log):
    w = workloads.make_rerank(2, 4096, seed=80, deep=True)
    run_and_check(w["parent"], w["confidence"], 100, exception_log)
    w = workloads.make_rerank(4, 500, seed=81, width=3, levels=4)  # many equal values
    for m in (7, 250):
        run_and_check(w["parent"], w["confidence"], m, exception_log)


def test_rerank_bad_trees_and_clamped_confidences(exception_log):
    w = workloads.make_rerank(5, 40, seed=82)
    par, conf = w["parent"].copy(), w["confidence"].copy()
    par[0, 0] = 0            # root with a parent
    par[1, 7] = 9            # a forward link
    conf[2, 5] = np.nan
    conf[3, 6] = 1.5
    conf[4, 0] = -0.25       # the root clamped to 0: every value is 0
    run_and_check(par, conf, 12, exception_log)


def test_rerank_output_feeds_tree_mask(exception_log):
    import speculative_decoding_verification_temp_gb300 as sv
    w = workloads.make_rerank(3, 300, seed=83)
    r = run_and_check(w["parent"], w["confidence"], 48, exception_log)
    mk = sv.tree_mask(r.parent, 64)
    torch.cuda.synchronize()
    for t in range(3):
        mw, pw, fw = ov.tree_mask(r.parent[t].cpu().numpy(), 64)
        assert fw == 0
        assert np.array_equal(mk.mask[t].cpu().numpy().view(np.uint64), mw)
