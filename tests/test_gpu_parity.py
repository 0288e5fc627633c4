"""CUDA path vs the CPU oracle, element by element, on seeded synthetic inputs.

Covers the five measured workloads at full size, the residual output, many
seeds, the pages' reference-function cases, and the edge cases (ragged and
tiny vocabularies, gamma 0 and 31, greedy rows, non-finite rows, bad tokens,
q(x) = 0, unaligned rows, top-k ties, chain/star/duplicate-token trees,
invalid and too-deep trees), plus a chi-square test of the GPU sampler.
"""

import numpy as np
import pytest
import scipy.stats
import torch

import speculative_decoding_verification_temp_gb300 as sv
from gpu_helpers import (compare_chain, compare_tree, oracle_chain, oracle_tree, run_chain,
                         run_tree, to_dev)
from oracle import philox
from oracle import verify as ov
from speculative_decoding_verification_temp_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()


# ---------------------------------------------------------------------------
# the five workloads at full size (the bench's launch configuration)
# ---------------------------------------------------------------------------

# "stream": no top-k array: chains of gamma <= 31 take the streaming chain path
# (rows, draw and precise kernels), trees of at most 256 nodes the tree walk
# (rows and walk kernels), longer chains and larger trees the streaming
# kernel; "resident": an all-off top-k array selects the resident cluster
# kernel on the same inputs.
PATHS = ["stream", "resident"]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("cfg", [0, 1, 2, 3])
def test_chain_workload_full_size(cfg, path, exception_log):
    w = workloads.config(cfg)
    res = run_chain(w, force_resident=path == "resident")
    compare_chain(res, oracle_chain(w), exception_log, f"config{cfg}-{path}", w["dtype"])


@pytest.mark.parametrize("path", PATHS)
def test_tree_workload_full_size(path, exception_log):
    w = workloads.config(4)
    assert w["parent"].shape == (32, 60) and w["max_depth"] == 6
    res = run_tree(w, force_resident=path == "resident")
    compare_tree(res, oracle_tree(w), exception_log, f"config4-{path}", w["dtype"])


def test_tree_mask_workload(exception_log):
    w = workloads.config(4)
    m = sv.tree_mask(torch.from_numpy(w["parent"]).cuda(), w["max_depth"])
    torch.cuda.synchronize()
    for t in range(w["parent"].shape[0]):
        mw, pw, fw = ov.tree_mask(w["parent"][t], w["max_depth"])
        np.testing.assert_array_equal(m.mask[t].cpu().numpy().view(np.uint64), mw)
        np.testing.assert_array_equal(m.position[t].cpu().numpy(), pw)
        assert int(m.flags[t]) == fw


# ---------------------------------------------------------------------------
# residual output, seeds, Philox
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("cfg", [0, 1])
def test_chain_residual_output(cfg, exception_log):
    w = workloads.config(cfg)
    res = run_chain(w, return_residual=True)
    compare_chain(res, oracle_chain(w), exception_log, f"resid{cfg}", w["dtype"],
                  check_residual=True)


@pytest.mark.parametrize("cfg,path", [(2, "stream"), (2, "resident"), (3, "resident")])
def test_chain_residual_output_full_size(cfg, path, exception_log):
    # every sequence of the full batch, in the bench's launch configuration:
    # the B = 256, V = 128256 workload on both kernels (residual within 2e-3
    # in bf16), and the V = 152064 workload with top-k 50 and 64 greedy rows
    w = workloads.config(cfg)
    res = run_chain(w, return_residual=True, force_resident=path == "resident")
    compare_chain(res, oracle_chain(w), exception_log, f"resid{cfg}-{path}", w["dtype"],
                  check_residual=True)


def test_tree_residual_output(exception_log):
    w = workloads.make_tree(16, 40, 8192, dtype="bf16", seed=5, branching=(4, 3, 2, 2, 1))
    res = run_tree(w, return_residual=True)
    compare_tree(res, oracle_tree(w), exception_log, "tree-resid", "bf16", check_residual=True)


@pytest.mark.parametrize("seed", range(12))
def test_chain_many_seeds(seed, exception_log):
    w = workloads.make_chain(64, 5, 32000, dtype="bf16", scale=2.0, zipf=1.1, sigma=0.7,
                             temperature=0.8, seed=20_000 + seed)
    res = run_chain(w, seed=seed)
    compare_chain(res, oracle_chain(w, seed=seed), exception_log, f"seed{seed}")


def test_override_equals_philox():
    """Passing the oracle's Philox uniforms as overrides reproduces the seeded run."""
    w = workloads.make_chain(32, 6, 5000, dtype="bf16", seed=3)
    B, G = 32, 7
    ov_u = np.zeros((B, G, 2), np.float32)
    for b in range(B):
        for i in range(G):
            for d in range(2):
                ov_u[b, i, d] = philox.uniform(w["seed"], b, i, d)
    a = run_chain(w)
    b = run_chain(w, uniform_override=ov_u)
    assert torch.equal(a.tokens, b.tokens) and torch.equal(a.num_accepted, b.num_accepted)


def test_repeated_calls_share_workspace():
    w1 = workloads.make_chain(16, 3, 3000, dtype="f32", seed=1)
    w2 = workloads.make_chain(8, 9, 3000, dtype="f32", seed=2)
    a1 = run_chain(w1)
    run_chain(w2)
    a2 = run_chain(w1)
    assert torch.equal(a1.tokens, a2.tokens) and torch.equal(a1.flags, a2.flags)


def test_workspace_needs_no_initialisation(exception_log):
    """Every call clears what must start at zero: a workspace full of 0xFF
    bytes, shared by calls of different shapes (whose layouts overlap each
    other's regions), still gives the oracle's results."""
    ws = torch.full((64 << 20,), 0xFF, dtype=torch.uint8, device="cuda")
    tw = workloads.make_tree(8, 30, 8192, dtype="bf16", seed=11, branching=(4, 3, 2, 1))
    c1 = workloads.make_chain(96, 7, 32000, dtype="bf16", seed=12, greedy_seqs=4)
    c2 = workloads.make_chain(8, 2, 32000, dtype="bf16", seed=13)
    c3 = workloads.make_chain(8, 3, 3001, dtype="f32", seed=14, top_k=20)
    for w in (tw, c1, c2, tw, c3, c1):
        if w["kind"] == "tree":
            compare_tree(run_tree(w, workspace_tensor=ws), oracle_tree(w), exception_log,
                         "dirty-ws-tree", w["dtype"])
        else:
            compare_chain(run_chain(w, workspace_tensor=ws), oracle_chain(w), exception_log,
                          "dirty-ws-chain", w["dtype"])


# ---------------------------------------------------------------------------
# the pages' reference-function cases, through logits
# ---------------------------------------------------------------------------

def prob_chain(p, q, token, u_accept, u_draw):
    """A one-draft chain whose rows are log-probabilities (T = 1)."""
    with np.errstate(divide="ignore"):
        lp = np.log(np.asarray(p, np.float64)).astype(np.float32)
        lq = np.log(np.asarray(q, np.float64)).astype(np.float32)
    target = np.stack([lp, np.zeros_like(lp)])[None]
    draft = lq[None, None]
    w = dict(dtype="f32", target=target, draft=draft, tokens=np.array([[token]], np.int32),
             target_temperature=np.ones(1, np.float32), draft_temperature=np.ones(1, np.float32),
             seed=0)
    uo = np.array([[[u_accept, u_draw], [0.0, 0.5]]], np.float32)
    return w, uo


@pytest.mark.parametrize("case", [
    ([0.8, 0.2], [0.2, 0.8], 1, 0.9, False, [1.0, 0.0]),
    ([0.8, 0.2], [0.8, 0.2], 0, 0.999, True, None),
    ([0.0, 1.0], [1.0, 0.0], 0, 0.0, False, [0.0, 1.0]),
])
def test_reference_function_cases(case, exception_log):
    p, q, tok, u, accepted, residual = case
    w, uo = prob_chain(p, q, tok, u, 0.5)
    res = run_chain(w, uniform_override=uo, return_residual=True)
    assert int(res.num_accepted[0]) == (1 if accepted else 0)
    if residual is not None:
        np.testing.assert_allclose(res.residual[0].cpu().numpy(), residual, atol=1e-6)
        assert int(res.tokens[0, 0]) == int(np.argmax(residual))
    compare_chain(res, oracle_chain(w, uniform_override=uo), exception_log, "page-asserts", "f32",
                  check_residual=True)


# ---------------------------------------------------------------------------
# edge cases
# ---------------------------------------------------------------------------

def random_chain(rng, B, gamma, V, dtype, ninf=0.0, temps=(1.0,), topks=(0,), scale=2.0):
    target = (rng.standard_normal((B, gamma + 1, V)) * scale).astype(np.float32)
    draft = (target[:, :gamma] + rng.standard_normal((B, gamma, V)) * 0.6).astype(np.float32)
    if ninf:
        target[rng.random(target.shape) < ninf] = -np.inf
        draft[rng.random(draft.shape) < ninf] = -np.inf
    if dtype == "bf16":
        workloads.round_bf16_inplace(target)
        workloads.round_bf16_inplace(draft)
    tokens = rng.integers(0, V, (B, gamma)).astype(np.int32)
    return dict(dtype=dtype, target=target, draft=draft, tokens=tokens,
                target_temperature=rng.choice(temps, B).astype(np.float32),
                draft_temperature=rng.choice(temps, B).astype(np.float32),
                target_top_k=rng.choice(topks, B).astype(np.int32),
                draft_top_k=rng.choice(topks, B).astype(np.int32), seed=int(rng.integers(1 << 40)))


@pytest.mark.parametrize("V", [1, 2, 3, 7, 8, 9, 33, 64, 65, 1000, 4099])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_small_and_ragged_vocab(V, dtype, exception_log):
    rng = np.random.default_rng(V * 7 + (dtype == "bf16"))
    for gamma in (0, 1, 3):
        w = random_chain(rng, 24, gamma, V, dtype, ninf=0.1, temps=(0.0, 0.5, 1.0, 2.0),
                         topks=(0, 1, 2, 5))
        # drafts drawn from the draft row where possible so that many are accepted
        for b in range(24):
            for i in range(gamma):
                if rng.random() < 0.7:
                    w["tokens"][b, i] = workloads.gumbel_argmax(rng, np.nan_to_num(
                        w["draft"][b, i], neginf=-1e30), 1.0)
        res = run_chain(w, return_residual=True)
        compare_chain(res, oracle_chain(w), exception_log, f"V{V}-{dtype}-g{gamma}", dtype,
                      check_residual=True)


@pytest.mark.parametrize("gamma", [0, 1, 31, 40])
def test_gamma_extremes(gamma, exception_log):
    w = workloads.make_chain(8, gamma, 2048, dtype="bf16", sigma=0.1, seed=gamma)
    res = run_chain(w)
    compare_chain(res, oracle_chain(w), exception_log, f"gamma{gamma}")


def test_all_greedy_rows(exception_log):
    w = workloads.make_chain(32, 4, 4000, dtype="bf16", seed=9, greedy_seqs=32)
    # some drafts differ from the argmax, ties at the max in a few rows
    w["tokens"][::3, 1] = 7
    w["target"][0, 0, :5] = w["target"][0, 0].max() + 1.0
    res = run_chain(w, return_residual=True)
    compare_chain(res, oracle_chain(w), exception_log, "greedy", check_residual=True)


def test_greedy_on_one_side_only(exception_log):
    w = workloads.make_chain(32, 3, 3000, dtype="f32", seed=10)
    w["draft_temperature"][:16] = 0.0  # greedy draft, sampled target
    w["target_temperature"][16:] = 0.0  # greedy target, sampled draft
    for b in range(16):
        for i in range(3):
            w["tokens"][b, i] = int(np.argmax(w["draft"][b, i]))
    res = run_chain(w, return_residual=True)
    compare_chain(res, oracle_chain(w), exception_log, "one-side-greedy", "f32",
                  check_residual=True)


def test_nonfinite_rows(exception_log):
    w = workloads.make_chain(12, 3, 600, dtype="f32", seed=11)
    w["target"][0, 0, 17] = np.nan
    w["target"][1, 1, 3] = np.inf
    w["draft"][2, 0, 5] = np.nan
    w["draft"][3, 0, :] = -np.inf
    w["target"][4, 0, :] = -np.inf
    w["target_temperature"][5] = -1.0
    w["draft_temperature"][6] = np.nan
    w["target_temperature"][7] = np.inf
    w["target"][8, 0, :] = np.nan
    res = run_chain(w, return_residual=True)
    flags = res.flags.cpu().numpy()
    assert all(flags[b] & sv.FLAG_NONFINITE for b in (0, 2, 3, 4, 5, 6, 7, 8))
    compare_chain(res, oracle_chain(w), exception_log, "nonfinite", "f32", check_residual=True)


def test_bad_tokens_and_zero_q(exception_log):
    w = workloads.make_chain(12, 3, 500, dtype="bf16", seed=12)
    w["tokens"][0, 0] = -1
    w["tokens"][1, 1] = 500
    w["tokens"][2, 2] = 10 ** 9
    for b in (3, 4, 5):
        w["draft"][b, 0, w["tokens"][b, 0]] = -np.inf  # q(x) = 0
    w["draft"][6, 0] = w["target"][6, 0]  # p = q with a forced rejection: degenerate residual
    w["tokens"][6, 0] = -5
    res = run_chain(w, return_residual=True)
    flags = res.flags.cpu().numpy()
    assert flags[0] & sv.FLAG_BAD_TOKEN and flags[3] & sv.FLAG_ZERO_Q
    assert flags[6] & sv.FLAG_DEGENERATE_RESIDUAL
    compare_chain(res, oracle_chain(w), exception_log, "bad-tokens", check_residual=True)


@pytest.mark.parametrize("dtype,pad", [("f32", 1), ("f32", 3), ("bf16", 1), ("bf16", 5)])
def test_unaligned_rows_take_scalar_path(dtype, pad, exception_log):
    w = workloads.make_chain(16, 3, 1001, dtype=dtype, seed=13 + pad)
    res = run_chain(w, pad_to=1001 + pad, return_residual=True)
    compare_chain(res, oracle_chain(w), exception_log, f"unaligned-{dtype}-{pad}", dtype,
                  check_residual=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_topk_with_ties(dtype, exception_log):
    rng = np.random.default_rng(14)
    B, gamma, V = 32, 3, 3001
    w = random_chain(rng, B, gamma, V, dtype, temps=(0.7, 1.0), topks=(1, 2, 3, 10, 50, 3000))
    w["target"] = np.round(w["target"] * 2) / 2  # coarse values: many ties at the threshold
    w["draft"] = np.round(w["draft"] * 2) / 2
    for b in range(B):
        for i in range(gamma):
            w["tokens"][b, i] = int(np.argmax(w["draft"][b, i]))
    res = run_chain(w, return_residual=True)
    compare_chain(res, oracle_chain(w), exception_log, f"topk-ties-{dtype}", dtype,
                  check_residual=True)


def test_mixed_policies_workload_residual(exception_log):
    w = workloads.make_chain(32, 4, 20000, dtype="bf16", seed=15, greedy_seqs=12, top_k=50,
                             temperature=0.7)
    res = run_chain(w, return_residual=True)
    compare_chain(res, oracle_chain(w), exception_log, "mixed", check_residual=True)


# ---------------------------------------------------------------------------
# trees
# ---------------------------------------------------------------------------

def tree_from_parents(parents, V, T=8, dtype="bf16", seed=0, dup=False, temperature=1.0):
    w = workloads.make_tree(T, len(parents), V, dtype=dtype, seed=seed, parents=parents,
                            temperature=temperature)
    depth = [0] * len(parents)
    for n in range(1, len(parents)):
        depth[n] = depth[parents[n]] + 1
    w["max_depth"] = max(depth)
    if dup:
        for t in range(T):
            for n in range(2, len(parents)):
                if parents[n] == parents[n - 1]:
                    w["tokens"][t, n] = w["tokens"][t, n - 1]
    return w


@pytest.mark.parametrize("shape", ["chain", "star", "dup", "binary", "single"])
def test_tree_shapes(shape, exception_log):
    if shape == "chain":
        parents = [-1] + list(range(7))
    elif shape == "star":
        parents = [-1] + [0] * 15
    elif shape == "dup":
        parents = [-1, 0, 0, 0, 1, 1, 2, 2, 3]
    elif shape == "binary":
        parents = [-1] + [(n - 1) // 2 for n in range(1, 31)]
    else:
        parents = [-1]
    w = tree_from_parents(parents, 64 if shape != "single" else 300, seed=len(parents),
                          dup=shape == "dup")
    res = run_tree(w, return_residual=True)
    compare_tree(res, oracle_tree(w), exception_log, f"tree-{shape}", check_residual=True)


def test_tree_small_vocab_many_rejections(exception_log):
    # a tiny vocabulary with a noisy draft forces many sibling rejections
    w = workloads.make_tree(64, 40, 16, dtype="f32", seed=16, sigma=2.0,
                            branching=(6, 3, 2, 1))
    res = run_tree(w, return_residual=True)
    compare_tree(res, oracle_tree(w), exception_log, "tree-smallV", "f32", check_residual=True)


def test_tree_greedy_and_topk(exception_log):
    w = workloads.make_tree(16, 30, 5000, dtype="bf16", seed=17, branching=(3, 3, 2, 1))
    w["target_temperature"][:8] = 0.0
    w["target_top_k"][8:] = 20
    w["draft_top_k"][8:] = 20
    res = run_tree(w, return_residual=True)
    compare_tree(res, oracle_tree(w), exception_log, "tree-greedy-topk", check_residual=True)


def test_invalid_and_deep_trees(exception_log):
    w = workloads.make_tree(4, 10, 256, dtype="bf16", seed=18, branching=(2, 2, 2, 2))
    w["parent"][0, 5] = 7   # parent after child
    w["parent"][1, 0] = 0   # root with a parent
    w["parent"][2, 3] = -4  # negative link
    w["max_depth"] = 2      # tree 3 is deeper than 2
    res = run_tree(w)
    flags = res.flags.cpu().numpy()
    assert flags[0] == sv.FLAG_BAD_TREE and flags[1] == sv.FLAG_BAD_TREE
    assert flags[2] == sv.FLAG_BAD_TREE and flags[3] == sv.FLAG_DEPTH
    assert (res.num_accepted.cpu().numpy() == -1).all()
    compare_tree(res, oracle_tree(w), exception_log, "tree-invalid")
    m = sv.tree_mask(torch.from_numpy(w["parent"]).cuda(), w["max_depth"])
    torch.cuda.synchronize()
    for t in range(4):
        mw, pw, fw = ov.tree_mask(w["parent"][t], w["max_depth"])
        np.testing.assert_array_equal(m.mask[t].cpu().numpy().view(np.uint64), mw)
        np.testing.assert_array_equal(m.position[t].cpu().numpy(), pw)
        assert int(m.flags[t]) == fw


@pytest.mark.parametrize("N", [1, 2, 63, 64, 65, 130, 1000, 4096])
def test_tree_mask_sizes(N):
    rng = np.random.default_rng(N)
    T = 3
    parent = np.zeros((T, N), np.int32)
    for t in range(T):
        parent[t, 0] = -1
        for n in range(1, N):
            parent[t, n] = int(rng.integers(max(0, n - 8), n))  # bounded depth growth
    m = sv.tree_mask(torch.from_numpy(parent).cuda(), 10 ** 6)
    torch.cuda.synchronize()
    for t in range(T):
        mw, pw, fw = ov.tree_mask(parent[t], 10 ** 6)
        np.testing.assert_array_equal(m.mask[t].cpu().numpy().view(np.uint64), mw)
        np.testing.assert_array_equal(m.position[t].cpu().numpy(), pw)
        assert int(m.flags[t]) == fw


# ---------------------------------------------------------------------------
# the GPU sampler's law
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("V", [4, 6, 8])
def test_first_token_law_chi_square(V):
    """Over many Philox keys the first output token follows p (chi-square)."""
    rng = np.random.default_rng(V)
    zp = rng.standard_normal(V).astype(np.float32)
    zq = (zp + rng.standard_normal(V) * 0.8).astype(np.float32)
    B, gamma = 200_000, 2
    target = np.broadcast_to(np.stack([zp] * (gamma + 1))[None], (B, gamma + 1, V)).copy()
    draft = np.broadcast_to(np.stack([zq] * gamma)[None], (B, gamma, V)).copy()
    q = np.exp(zq.astype(np.float64) - zq.max())
    q /= q.sum()
    tokens = rng.choice(V, size=(B, gamma), p=q).astype(np.int32)
    res = sv.verify_chain(to_dev(target, "f32"), to_dev(draft, "f32"),
                          torch.from_numpy(tokens).cuda(), 1.0, 1.0, seed=987654321)
    first = res.tokens[:, 0].cpu().numpy()
    p = np.exp(zp.astype(np.float64) - zp.max())
    p /= p.sum()
    counts = np.bincount(first, minlength=V)
    stat, pval = scipy.stats.chisquare(counts, B * p)
    assert pval > 1e-6, (counts, B * p, pval)
