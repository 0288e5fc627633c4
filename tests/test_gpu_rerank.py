"""EAGLE-2 rerank on the GPU against the oracle: kept nodes, re-indexed
parents, counts and flags bit-exact, values equal (both sides take the same
float32 products in the same order)."""

import numpy as np
import pytest
import torch

from oracle import verify as ov
from speculative_decoding_verification_temp_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()


def run_and_check(parent, conf, m):
    import speculative_decoding_verification_temp_gb300 as sv
    r = sv.tree_rerank(torch.from_numpy(parent).cuda(), torch.from_numpy(conf).cuda(), m)
    torch.cuda.synchronize()
    nodes, newp, val = r.nodes.cpu().numpy(), r.parent.cpu().numpy(), r.value.cpu().numpy()
    count, flags = r.count.cpu().numpy(), r.flags.cpu().numpy()
    for t in range(parent.shape[0]):
        wn, wp, wv, wf = ov.tree_rerank(parent[t], conf[t], m)
        k = len(wn)
        assert count[t] == k and flags[t] == wf, (t, count[t], k, flags[t], wf)
        assert list(nodes[t, :k]) == wn and list(newp[t, :k]) == wp
        assert np.array_equal(val[t, :k], np.asarray(wv, np.float32))
        assert (nodes[t, k:] == -1).all() and (newp[t, k:] == -1).all()
    return r


@pytest.mark.parametrize("N", [1, 2, 17, 60, 1000, 4096])
def test_rerank_random_trees(N):
    w = workloads.make_rerank(6, N, seed=70 + N)
    for m in sorted({1, 5, 64, N, N + 3}):
        run_and_check(w["parent"], w["confidence"], m)


def test_rerank_deep_chain_and_coarse_ties():
    w = workloads.make_rerank(2, 4096, seed=80, deep=True)
    run_and_check(w["parent"], w["confidence"], 100)
    w = workloads.make_rerank(4, 500, seed=81, width=3, levels=4)  # many equal values
    for m in (7, 250):
        run_and_check(w["parent"], w["confidence"], m)


def test_rerank_bad_trees_and_clamped_confidences():
    w = workloads.make_rerank(5, 40, seed=82)
    par, conf = w["parent"].copy(), w["confidence"].copy()
    par[0, 0] = 0            # root with a parent
    par[1, 7] = 9            # a forward link
    conf[2, 5] = np.nan
    conf[3, 6] = 1.5
    conf[4, 0] = -0.25       # the root clamped to 0: every value is 0
    run_and_check(par, conf, 12)


def test_rerank_output_feeds_tree_mask():
    import speculative_decoding_verification_temp_gb300 as sv
    w = workloads.make_rerank(3, 300, seed=83)
    r = run_and_check(w["parent"], w["confidence"], 48)
    mk = sv.tree_mask(r.parent, 64)
    torch.cuda.synchronize()
    for t in range(3):
        mw, pw, fw = ov.tree_mask(r.parent[t].cpu().numpy(), 64)
        assert fw == 0
        assert np.array_equal(mk.mask[t].cpu().numpy().view(np.uint64), mw)
