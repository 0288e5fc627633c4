"""GB300-native speculative-sampling verification.

The computation lives in libspecverify.so (CUDA for sm_103a, C ABI declared
in include/specverify.h); ``api`` is a thin torch binding over it.

  verify_chain   accept drafts with probability min(1, p/q), stop at the first
                 rejection, draw the correction from norm([p - q]+) or a bonus
                 token from p
  verify_tree    recursive rejection over sibling candidates of token trees
  tree_mask      ancestor-or-self attention masks and depth position ids
  overlap        per-position acceptance rate beta_i = sum_v min(p_i, q_i)
  typical_accept typical acceptance (entropy threshold; approximate, not
                 distribution-exact)
  tree_rerank    EAGLE-2 rerank: the top-m nodes of a draft tree by path value
"""

from ._abi import (FLAG_BAD_TOKEN, FLAG_BAD_TREE, FLAG_DEGENERATE_RESIDUAL, FLAG_DEPTH,  # noqa: F401
                   FLAG_NONFINITE, FLAG_TIMEOUT, FLAG_ZERO_Q)


def __getattr__(name):
    # the torch binding is imported on first use, so the workload generator
    # and the build step do not need torch
    if name in ("verify_chain", "verify_chain_static", "verify_tree", "tree_mask", "overlap",
                "typical_accept", "tree_rerank", "SpecVerifyError", "workspace",
                "ChainResult", "TreeResult", "MaskResult", "OverlapResult", "TypicalResult",
                "RerankResult", "set_wait_limit", "api"):
        import importlib
        api = importlib.import_module(__name__ + ".api")
        return api if name == "api" else getattr(api, name)
    raise AttributeError(name)
