"""The tree walk over the rows stream (aligned rows, at most 256 nodes, no row
filter) against the oracle, on the cases its design singles out.

- more children at a node than a warp has lanes, the largest tree it takes
  (256 nodes) and the first one it does not (257 nodes: the streaming
  kernel);
- a degenerate residual: p = q with children whose tokens are rejected for a
  bad token, so that every residual pass has total 0 and the draw falls back
  to the held p;
- a greedy draft (one-hot q: q(x) = 0 off its argmax) and a greedy target;
- non-finite target and draft rows on the path;
- a bounded wait of the rows kernel that runs out (the documented fallback),
  and the next call bit-exact with one made before;
- rows whose per-CTA share does not fit the staging buffer (the passes then
  read global memory).
"""

import numpy as np
import pytest
import torch

from gpu_helpers import compare_tree, oracle_tree, run_tree
from speculative_decoding_verification_temp_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()


def star(n_children, depth_tail=0):
    """Root with n_children children, the last of which heads a chain of
    depth_tail more nodes."""
    parents = [-1] + [0] * n_children
    last = n_children
    for _ in range(depth_tail):
        parents.append(last)
        last = len(parents) - 1
    return parents


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_many_children(dtype, exception_log):
    # 40 children at the root with a noisy draft: most are rejected in turn
    w = workloads.make_tree(12, 44, 300, dtype=dtype, seed=301, sigma=2.5,
                            parents=star(40, depth_tail=3), branching=(1,) * 4)
    res = run_tree(w, return_residual=True)
    compare_tree(res, oracle_tree(w), exception_log, f"walk-star40-{dtype}", dtype,
                 check_residual=True)


@pytest.mark.parametrize("N", [255, 256, 257])
def test_largest_trees(N, exception_log):
    # 256 nodes is the walk's limit; 257 takes the streaming kernel
    w = workloads.make_tree(3, N, 4000, dtype="bf16", seed=N, sigma=1.0,
                            branching=(6, 4, 3, 2, 2, 1, 1))
    assert w["parent"].shape == (3, N)
    res = run_tree(w, return_residual=True)
    compare_tree(res, oracle_tree(w), exception_log, f"walk-N{N}", "bf16", check_residual=True)


def test_degenerate_residual(exception_log):
    # p = q: every residual total is 0; children with out-of-range tokens are
    # rejected (bad token), each rejection flags the residual degenerate and
    # the held p stays; the last child is valid and accepted, or the draw
    # falls back to p
    w = workloads.make_tree(6, 8, 512, dtype="f32", seed=302, sigma=0.0,
                            parents=[-1, 0, 0, 0, 1, 1, 4, 4], branching=(1, 1, 1))
    w["draft"] = w["target"].copy()
    w["tokens"][:, 1] = -1
    w["tokens"][:, 2] = 512
    w["tokens"][:3, 3] = -7  # trees 0-2: every child of the root is bad
    w["tokens"][:, 4] = 10**6
    res = run_tree(w, return_residual=True)
    want = oracle_tree(w)
    # the oracle flags the bad tokens and the degenerate residual
    assert all(r["flags"] & 1 and r["flags"] & 8 for r in want)
    compare_tree(res, want, exception_log, "walk-degenerate", "f32", check_residual=True)


def test_greedy_draft_and_target(exception_log):
    w = workloads.make_tree(16, 30, 3000, dtype="bf16", seed=303, sigma=0.7,
                            branching=(3, 3, 2, 1))
    w["draft_temperature"][:6] = 0.0   # one-hot q
    w["target_temperature"][6:11] = 0.0  # greedy target
    w["draft_temperature"][11:] = 0.6
    w["target_temperature"][11:] = 1.3
    res = run_tree(w, return_residual=True)
    compare_tree(res, oracle_tree(w), exception_log, "walk-greedy", "bf16", check_residual=True)


def test_nonfinite_rows(exception_log):
    w = workloads.make_tree(5, 12, 2000, dtype="f32", seed=304, sigma=0.5, branching=(3, 2, 2))
    w["target"][0, 0, 17] = np.nan          # root target row NaN
    w["draft"][1, 0, 5] = np.inf            # root draft row +inf
    w["target"][2, 0, :] = -np.inf          # root target row with no finite entry
    w["target"][3, 0, 100:] = -np.inf       # masked tail, still a valid distribution
    w["draft"][4, 0, :] = -np.inf           # root draft row with no finite entry
    res = run_tree(w, return_residual=True)
    compare_tree(res, oracle_tree(w), exception_log, "walk-nonfinite", "f32", check_residual=True)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_wait_runs_out_then_recovers(dtype):
    import speculative_decoding_verification_temp_gb300 as sv
    w = workloads.make_tree(4, 20, 50000, dtype=dtype, seed=305, branching=(3, 2, 2, 1))

    def call():
        r = run_tree(w, return_residual=True)
        return [x.cpu().numpy() for x in (r.num_accepted, r.path, r.tokens, r.flags, r.residual)]

    before = call()
    assert not np.any(before[3] & sv.FLAG_TIMEOUT)
    try:
        sv.set_wait_limit(0)
        n, path, toks, flags, resid = call()
    finally:
        sv.set_wait_limit(None)
    assert np.all(n == 0)
    assert np.all(path == -1) and np.all(toks == -1)
    assert np.all(flags == sv.FLAG_TIMEOUT)
    assert np.all(resid == 0.0)
    after = call()
    for a, b in zip(before, after):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("dtype,V", [("f32", 100_000), ("bf16", 200_000)])
def test_rows_from_global_memory(dtype, V, exception_log):
    # a CTA's share of a row pair larger than its staging buffer: the passes
    # read the rows from global memory
    w = workloads.make_tree(3, 10, V, dtype=dtype, seed=306, sigma=1.2, branching=(3, 2, 1))
    res = run_tree(w, return_residual=True)
    compare_tree(res, oracle_tree(w), exception_log, f"walk-global-{dtype}", dtype,
                 check_residual=True)
