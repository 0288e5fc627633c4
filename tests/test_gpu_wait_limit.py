"""A bounded on-device wait that runs out, on purpose and without a fault.

Every wait inside the kernels gives up after a bound and reports
SPEC_FLAG_TIMEOUT instead of hanging.  spec_set_wait_limit shortens the chain
rows kernel's first wait on each chunk to a single non-blocking test, which
gives up whenever a chunk's copy has not landed yet (a copy of 32 KiB from
HBM takes longer than one test).  The kernel then waits again with the full
bound, so no copy is left in flight and the call completes.  The test checks
the documented fallback (0 accepted drafts, every token -1, flags exactly
SPEC_FLAG_TIMEOUT, a zero residual) and that the next call with the default
bound is bit-exact with a call made before.
"""

import numpy as np
import pytest
import torch

from gpu_helpers import to_dev
from speculative_decoding_verification_temp_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()


def call(sv, w, dt):
    r = sv.verify_chain(to_dev(w["target"], dt), to_dev(w["draft"], dt),
                        torch.from_numpy(w["tokens"]).cuda(), w["target_temperature"],
                        w["draft_temperature"], seed=w["seed"], return_residual=True)
    torch.cuda.synchronize()
    return [x.cpu().numpy() for x in r]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_first_wait_runs_out_then_recovers(dtype):
    import speculative_decoding_verification_temp_gb300 as sv
    w = workloads.make_chain(8, 4, 50000, dtype=dtype, seed=211)
    before = call(sv, w, dtype)
    assert not np.any(before[2] & sv.FLAG_TIMEOUT)
    try:
        sv.set_wait_limit(0)
        n, toks, flags, resid = call(sv, w, dtype)
    finally:
        sv.set_wait_limit(None)
    B, gamma = w["B"], w["draft"].shape[1]
    assert np.all(n == 0)
    assert np.all(toks == -1) and toks.shape == (B, gamma + 1)
    assert np.all(flags == sv.FLAG_TIMEOUT)
    assert np.all(resid == 0.0)
    after = call(sv, w, dtype)
    for a, b in zip(before, after):
        assert np.array_equal(a, b)
