"""spec_verify_chain_static (the entry point on the library's fixed scratch)
against spec_verify_chain (caller workspace) on the same inputs.

Both calls run the same verification kernels, so integer outputs must be
identical and residuals must agree within the parity tolerance of the logit
dtype.  Two static calls in a row check that a completed call leaves the
scratch ready for the next one.  This file is collected last so that it also
runs after every other GPU test in the same process.
"""

import numpy as np
import pytest
import torch

import speculative_decoding_verification_temp_gb300 as sv
from speculative_decoding_verification_temp_gb300 import _abi, workloads

from gpu_helpers import RESID_TOL, to_dev

pytestmark = pytest.mark.gpu


def _args(w):
    dt = w["dtype"]
    kp = w.get("target_top_k")
    kq = w.get("draft_top_k")
    return dict(
        target_logits=to_dev(w["target"], dt), draft_logits=to_dev(w["draft"], dt),
        draft_tokens=torch.from_numpy(w["tokens"]).cuda(),
        target_temperature=w["target_temperature"], draft_temperature=w["draft_temperature"],
        target_top_k=None if kp is None or not np.any(kp) else kp,
        draft_top_k=None if kq is None or not np.any(kq) else kq,
        seed=w["seed"], return_residual=True)


def _same(a, b, dtype):
    assert torch.equal(a.num_accepted, b.num_accepted)
    assert torch.equal(a.tokens, b.tokens)
    assert torch.equal(a.flags, b.flags)
    err = (a.residual - b.residual).abs().max().item()
    assert err <= RESID_TOL[dtype], err


@pytest.mark.parametrize("case", [
    # streaming chain path: bf16, aligned rows, no filters; 1024 units (the largest
    # B = 128, gamma = 7 batch that fits the scratch)
    dict(B=128, gamma=7, V=32000, dtype="bf16", greedy_seqs=8, top_k=0),
    # resident kernel: fp32 with top-k filtering
    dict(B=16, gamma=4, V=5000, dtype="f32", greedy_seqs=2, top_k=50),
])
def test_static_scratch_matches_workspace_entry(case):
    w = workloads.make_chain(seed=41, **case)
    args = _args(w)
    want = sv.verify_chain(**args)
    first = sv.verify_chain_static(**args)
    second = sv.verify_chain_static(**args)
    torch.cuda.synchronize()
    assert int((want.num_accepted >= 0).sum()) == case["B"]
    _same(first, want, case["dtype"])
    _same(second, want, case["dtype"])


def test_static_scratch_rejects_oversize_shapes():
    # 8192 sequences of 7 drafts need more workspace than the scratch holds,
    # even with a 64-entry vocabulary: refused with SPEC_ERR_UNSUPPORTED
    B, gamma, V = 8192, 7, 64
    lib = _abi.load()
    assert lib.spec_verify_chain_workspace_size(B, gamma, V, _abi.SPEC_BF16) > \
        _abi.SPEC_STATIC_SCRATCH_BYTES
    g = torch.Generator(device="cuda").manual_seed(3)
    target = torch.randn(B, gamma + 1, V, device="cuda", generator=g).to(torch.bfloat16)
    draft = torch.randn(B, gamma, V, device="cuda", generator=g).to(torch.bfloat16)
    tokens = torch.zeros(B, gamma, dtype=torch.int32, device="cuda")
    with pytest.raises(sv.SpecVerifyError, match="UNSUPPORTED"):
        sv.verify_chain_static(target, draft, tokens, 1.0, 1.0, seed=1)
