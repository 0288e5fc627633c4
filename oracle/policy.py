"""Sampling policy: logits -> the distribution that enters the acceptance rule.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  float64 throughout.

Pages followed
  whoami-wesleyyou.top "Speculative Decoding" notes, § 从 LM head 到 sampling
  distribution: the LM head gives logits z; temperature, softmax and top-k
  turn them into the sampling distribution; greedy decoding puts all mass on
  the argmax token; p and q may use different policies, but q must be the
  distribution the draft was actually drawn from.
  wineandchord.com "推测解码：接受规则、状态与收益边界", § 与 Logit Processor
  的组合: the acceptance ratio uses the processed p_i and q_i (temperature,
  top-k among the listed processors).
  tannlonggtaoo.github.io "Speculative Decoding", § Greedy Sampling:
  temperature 0 reduces verification to comparing against the argmax.

Readings where the pages are silent:
  * greedy / argmax tie-break: the lowest index among the maxima;
  * top-k selects on the raw logits (before temperature); the threshold is the
    k-th largest raw value and every entry >= threshold is kept, so ties at the
    threshold are all kept; k <= 0 or k >= V means no filtering;
  * a row is "non-finite" when the temperature is NaN, negative or infinite,
    or the logits hold a NaN or +inf, or no finite logit at all; such a row is
    flagged and replaced by the one-hot distribution at the finite argmax
    (index 0 when nothing is finite).  The pages only say such inputs are
    errors (verify_candidate raises ValueError on non-finite probabilities).
  * top-p and min-p: the pages list them among the processors p and q must
    share (wineandchord.com, § 与 Logit Processor 的组合) but define neither.  The plain published
    definitions are used: top-p (nucleus sampling, Holtzman et al., "The
    Curious Case of Neural Text Degeneration", ICLR 2020) keeps the smallest
    set of most probable tokens whose mass reaches p; min-p keeps the tokens
    whose probability is at least min_p times the largest.  Order: temperature
    and top-k, then top-p on that distribution, then min-p on the result, each
    renormalised.  Ties at a boundary value are all kept, as for top-k.
    top_p >= 1 and min_p <= 0 mean no filtering.  Where float rounding puts
    a cumulative mass within 1e-12 of p the decision is the float64 one here;
    a GPU decision in float32 may differ there (a parity excuse, not a pin).
"""

import numpy as np

FLAG_NONFINITE = 4


class Dist:
    """A policy result: either one-hot at ``index`` or a probability vector."""

    __slots__ = ("onehot", "index", "probs", "flags")

    def __init__(self, onehot, index=None, probs=None, flags=0):
        self.onehot = onehot
        self.index = index
        self.probs = probs
        self.flags = flags

    def dense(self, V, dtype=np.float64):
        """The distribution as a length-V vector."""
        if self.onehot:
            out = np.zeros(V, dtype=dtype)
            out[self.index] = 1
            return out
        return self.probs


def finite_argmax(z):
    """Lowest index of the largest finite logit; 0 when no logit is finite."""
    z = np.asarray(z, dtype=np.float64)
    finite = np.isfinite(z)
    if not finite.any():
        return 0
    best = z[finite].max()
    return int(np.flatnonzero(finite & (z == best))[0])


def topk_threshold(z, k):
    """k-th largest raw logit value (k counted from 1), or None for no filter."""
    V = z.shape[0]
    if k <= 0 or k >= V:
        return None
    ordered = np.sort(z)[::-1]
    return ordered[k - 1]


def policy_distribution(z, temperature, top_k=0):
    """Apply one row's policy (temperature T, top-k) to logits z.

    T == 0      -> greedy: one-hot at the argmax (lowest index on ties).
    T > 0       -> softmax(z / T) over the entries kept by top-k.
    bad input   -> one-hot at the finite argmax, flagged FLAG_NONFINITE.
    """
    z = np.asarray(z, dtype=np.float64)
    T = float(temperature)
    bad = (not np.isfinite(T)) or T < 0.0
    bad = bad or bool(np.isnan(z).any()) or bool(np.isposinf(z).any())
    bad = bad or not bool(np.isfinite(z).any())
    if bad:
        return Dist(True, index=finite_argmax(z), flags=FLAG_NONFINITE)
    if T == 0.0:
        return Dist(True, index=finite_argmax(z))
    thr = topk_threshold(z, int(top_k))
    kept = z if thr is None else np.where(z >= thr, z, -np.inf)
    m = kept.max()
    weights = np.exp((kept - m) / T)
    return Dist(False, probs=weights / weights.sum())


def topp_threshold(probs, top_p):
    """Smallest probability kept by top-p: the value at which the descending
    cumulative mass first reaches top_p (None for no filter).

    Out-of-range readings (the pages define neither filter): top_p >= 1 or NaN
    is no filter; top_p <= 0 keeps the most probable value (and its ties)."""
    top_p = float(top_p)
    if not top_p < 1.0:  # also NaN
        return None
    ordered = np.sort(np.asarray(probs, dtype=np.float64))[::-1]
    i = int(np.searchsorted(np.cumsum(ordered), top_p, side="left"))
    return ordered[min(i, len(ordered) - 1)]


def topp_filter(probs, top_p):
    """Nucleus (top-p) filtering of a probability vector, renormalised; every
    entry tied with the boundary value is kept."""
    probs = np.asarray(probs, dtype=np.float64)
    thr = topp_threshold(probs, top_p)
    if thr is None:
        return probs
    kept = np.where(probs >= thr, probs, 0.0)
    return kept / kept.sum()


def minp_filter(probs, min_p):
    """Min-p filtering: keep p(x) >= min_p * max p, renormalised.

    Out-of-range readings: min_p <= 0 or NaN is no filter; min_p > 1 is taken
    as 1 (only the most probable value and its ties are kept), so the kept
    mass is never empty."""
    probs = np.asarray(probs, dtype=np.float64)
    min_p = float(min_p)
    if not min_p > 0.0:  # also NaN
        return probs
    min_p = min(min_p, 1.0)
    kept = np.where(probs >= min_p * probs.max(), probs, 0.0)
    return kept / kept.sum()


def policy_distribution_ext(z, temperature, top_k=0, top_p=1.0, min_p=0.0):
    """policy_distribution followed by top-p and then min-p (see the module
    readings); a greedy or non-finite row stays one-hot."""
    d = policy_distribution(z, temperature, top_k)
    if d.onehot:
        return d
    probs = minp_filter(topp_filter(d.probs, top_p), min_p)
    return Dist(False, probs=probs, flags=d.flags)
