"""Per-position overlap beta_i = sum_v min(p_i(v), q_i(v)) on the GPU against
the oracle, element by element.

Tolerance: both sides read the same logit values (bf16 inputs are exact in
fp32 and float64); the GPU's error is its arithmetic: a relative error below
about 2e-7 per exponential and per normaliser, and sums kept in double-float
or double, so |beta_gpu - beta| stays below about 1e-6.  The test allows 1e-5.
"""

import numpy as np
import pytest
import torch

from gpu_helpers import to_dev
from oracle import verify as ov
from speculative_decoding_verification_temp_gb300 import workloads

pytestmark = pytest.mark.gpu

TOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()


def run(w, seqs=None, pad_to=None):
    import speculative_decoding_verification_temp_gb300 as sv
    t, d = w["target"], w["draft"]
    if pad_to is not None:
        V = t.shape[-1]
        tp = np.zeros(t.shape[:-1] + (pad_to,), np.float32)
        tp[..., :V] = t
        dp = np.zeros(d.shape[:-1] + (pad_to,), np.float32)
        dp[..., :V] = d
        td, dd = to_dev(tp, w["dtype"])[..., :V], to_dev(dp, w["dtype"])[..., :V]
    else:
        td, dd = to_dev(t, w["dtype"]), to_dev(d, w["dtype"])
    res = sv.overlap(td, dd, w["target_temperature"], w["draft_temperature"])
    torch.cuda.synchronize()
    return res.beta.cpu().numpy(), res.flags.cpu().numpy()


def want(w, seqs):
    return ov.chain_overlap(w["target"][seqs], w["draft"][seqs], w["target_temperature"][seqs],
                            w["draft_temperature"][seqs])


@pytest.mark.parametrize("cfg", [0, 1, 2])
def test_overlap_workloads(cfg):
    w = workloads.config(cfg)
    beta, flags = run(w)
    seqs = np.arange(min(w["B"], 24))  # the oracle on a prefix of the batch at full size
    ref = want(w, seqs)
    assert np.abs(beta[seqs] - ref).max() <= TOL
    assert (flags == 0).all()
    assert (beta >= 0).all() and (beta <= 1 + 1e-6).all()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_overlap_greedy_sides_and_ragged_vocab(dtype):
    rng = np.random.default_rng(41)
    B, gamma, V = 6, 3, 1001
    t = (2.0 * rng.standard_normal((B, gamma + 1, V))).astype(np.float32)
    d = (t[:, :gamma] + 0.3 * rng.standard_normal((B, gamma, V))).astype(np.float32)
    if dtype == "bf16":
        workloads.round_bf16_inplace(t)
        workloads.round_bf16_inplace(d)
    tt = np.array([1.0, 0.0, 1.0, 0.0, 0.7, 1.3], np.float32)
    td = np.array([1.0, 1.0, 0.0, 0.0, 0.7, 0.9], np.float32)
    w = dict(target=t, draft=d, target_temperature=tt, draft_temperature=td, dtype=dtype)
    beta, flags = run(w)
    ref = want(w, np.arange(B))
    assert np.abs(beta - ref).max() <= TOL
    # unaligned rows take the scalar path and give the same values
    beta_u, _ = run(w, pad_to=V + 3)
    assert np.abs(beta_u - ref).max() <= TOL


def test_overlap_nonfinite_rows_are_flagged():
    rng = np.random.default_rng(42)
    B, gamma, V = 4, 2, 512
    t = rng.standard_normal((B, gamma + 1, V)).astype(np.float32)
    d = (t[:, :gamma] + 0.2 * rng.standard_normal((B, gamma, V))).astype(np.float32)
    t[1, 0, 7] = np.nan
    d[2, 1, 9] = np.inf
    tt = np.ones(B, np.float32)
    td = np.ones(B, np.float32)
    td[3] = -1.0  # a negative temperature is not finite either
    w = dict(target=t, draft=d, target_temperature=tt, draft_temperature=td, dtype="f32")
    beta, flags = run(w)
    ref = want(w, np.arange(B))
    assert np.abs(beta - ref).max() <= TOL
    assert list(flags & 4) == [0, 4, 4, 4]


@pytest.mark.parametrize("V", [1, 5, 37])
def test_overlap_tiny_vocab_with_empty_slices(V):
    # a vocabulary shorter than the cluster's slices leaves the later slices empty
    rng = np.random.default_rng(43 + V)
    B, gamma = 3, 2
    t = rng.standard_normal((B, gamma + 1, V)).astype(np.float32)
    d = rng.standard_normal((B, gamma, V)).astype(np.float32)
    tt = np.array([1.0, 0.0, 0.6], np.float32)
    td = np.array([1.0, 0.8, 0.0], np.float32)
    w = dict(target=t, draft=d, target_temperature=tt, draft_temperature=td, dtype="f32")
    beta, flags = run(w)
    ref = want(w, np.arange(B))
    assert np.abs(beta - ref).max() <= TOL
    assert (flags == 0).all()


def test_overlap_greedy_ties_across_slices():
    # equal maxima in the first and the last slice: the greedy side is the
    # one-hot at the lower index
    rng = np.random.default_rng(44)
    B, gamma, V = 2, 2, 4099
    t = rng.standard_normal((B, gamma + 1, V)).astype(np.float32)
    d = rng.standard_normal((B, gamma, V)).astype(np.float32)
    for b in range(B):
        for i in range(gamma):
            t[b, i, [3, V - 2]] = 9.0
            d[b, i, [5, V - 1]] = 9.0
    tt = np.array([0.0, 1.0], np.float32)
    td = np.array([1.0, 0.0], np.float32)
    w = dict(target=t, draft=d, target_temperature=tt, draft_temperature=td, dtype="f32")
    beta, _ = run(w)
    ref = want(w, np.arange(B))
    assert np.abs(beta - ref).max() <= TOL


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_overlap_large_vocab(dtype):
    # 262147 entries: slices of 65544 entries per CTA of a cluster of 4, a
    # ragged last slice, rows that are not 16-byte aligned (element loads)
    rng = np.random.default_rng(45)
    B, gamma, V = 2, 2, 262147
    t = (3.0 * rng.standard_normal((B, gamma + 1, V))).astype(np.float32)
    d = (t[:, :gamma] + 0.5 * rng.standard_normal((B, gamma, V))).astype(np.float32)
    if dtype == "bf16":
        workloads.round_bf16_inplace(t)
        workloads.round_bf16_inplace(d)
    tt = np.array([1.0, 0.7], np.float32)
    td = np.array([1.0, 1.1], np.float32)
    w = dict(target=t, draft=d, target_temperature=tt, draft_temperature=td, dtype=dtype)
    beta, _ = run(w)
    ref = want(w, np.arange(B))
    assert np.abs(beta - ref).max() <= TOL


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_overlap_masked_vocab_and_hidden_nan(dtype):
    # -inf over half the vocabulary (a masked vocabulary); in sequence 1 a NaN
    # sits inside the masked half, where no finite logit shares its group
    rng = np.random.default_rng(46)
    B, gamma, V = 3, 2, 4096
    t = rng.standard_normal((B, gamma + 1, V)).astype(np.float32)
    d = (t[:, :gamma] + 0.4 * rng.standard_normal((B, gamma, V))).astype(np.float32)
    t[:, :, : V // 2] = -np.inf
    d[:, :, : V // 2] = -np.inf
    t[1, 0, 100] = np.nan
    if dtype == "bf16":
        workloads.round_bf16_inplace(t)
        workloads.round_bf16_inplace(d)
    tt = np.array([1.0, 1.0, 0.5], np.float32)
    td = np.array([1.0, 1.0, 0.8], np.float32)
    w = dict(target=t, draft=d, target_temperature=tt, draft_temperature=td, dtype=dtype)
    beta, flags = run(w)
    ref = want(w, np.arange(B))
    assert np.abs(beta - ref).max() <= TOL
    assert list(flags & 4) == [0, 4, 0]
