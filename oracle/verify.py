"""Speculative-sampling verification, written step by step from the pages.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The probability-level functions (``accept_test``, ``positive_residual``,
``inverse_cdf``, ``walk_chain``, ``walk_tree``) use only numpy operations that
also work on object arrays of ``fractions.Fraction``; the logit-level entry
points (``verify_chain``, ``verify_tree``) apply ``oracle.policy`` in float64
and then call them.

Flag bits are the interface values of the library's per-sequence flag word.
"""

import math

import numpy as np

from . import philox
from .policy import Dist, finite_argmax, policy_distribution, policy_distribution_ext

FLAG_BAD_TOKEN = 1
FLAG_ZERO_Q = 2
FLAG_NONFINITE = 4
FLAG_DEGENERATE_RESIDUAL = 8
FLAG_DEPTH = 16
FLAG_TIMEOUT = 32
FLAG_BAD_TREE = 64


# ---------------------------------------------------------------------------
# single position
# ---------------------------------------------------------------------------

def accept_test(p, q, x, u):
    """Accept draft token x iff u < alpha, alpha = min(1, p(x)/q(x)).

    whoami-wesleyyou.top "Speculative Decoding" notes, § Acceptance 与
    correction (boxed alpha(x) = min{1, p(x)/q(x)}); wineandchord.com
    "推测解码：接受规则、状态与收益边界", § 单位置接受 reference (the test is
    ``uniform < accept_probability`` with uniform in [0, 1), and a draft token
    with q(token) <= 0 or outside the vocabulary is an error there).

    The pages write the comparison both as U <= alpha and as u < alpha; the
    strict form is the one the reference function's assert forces (p(x) = 0,
    u = 0 must reject).  Errors become flags and a rejection here.

    Returns (accepted, alpha, flags).  Parity: pinned (page asserts, worked
    examples, exact enumeration).
    """
    V = len(p)
    if not (0 <= int(x) < V):
        return False, 0, FLAG_BAD_TOKEN
    qx = q[int(x)]
    if not qx > 0:
        return False, 0, FLAG_ZERO_Q
    alpha = min(1, p[int(x)] / qx)
    return bool(u < alpha), alpha, 0


def positive_residual(p, q):
    """r = [p - q]_+ / Z with Z = sum [p - q]_+.

    whoami-wesleyyou.top "Speculative Decoding" notes, § Correction 为什么用正
    残差 (r(x) = [p(x) - q(x)]_+ / Z, Z = 1 - beta); wineandchord.com
    "推测解码：接受规则、状态与收益边界", § 正确性契约 (clamp negatives before
    normalising; a degenerate residual sum needs a defined fallback).

    Returns (r, Z, flags); when Z <= 0, r is None and FLAG_DEGENERATE_RESIDUAL
    is set (the caller keeps the distribution it had: our reading of the
    fallback the pages ask for).  Parity: pinned (worked examples A and B,
    exact enumeration).
    """
    w = np.maximum(p - q, 0)
    Z = w.sum()
    if not Z > 0:
        return None, Z, FLAG_DEGENERATE_RESIDUAL
    return w / Z, Z, 0


def inverse_cdf(weights, u):
    """Draw one token from non-negative ``weights`` with the uniform u.

    The pages only say "sample from" a distribution.  Reading (parity
    unpinned by the pages; pinned oracle<->GPU): inverse CDF in index order,
    token = smallest v with sum_{w<=v} weights_w > u * sum_w weights_w; if
    rounding leaves no such v, the largest v with weights_v > 0.  A token
    with zero weight is never returned.

    Returns (token, margin): margin is the distance from u to the nearer
    normalised CDF boundary around the returned token (0 on the fallback),
    used to excuse GPU disagreements that lie within rounding of a boundary.
    """
    c = np.cumsum(weights)
    total = c[-1]
    t = u * total
    above = np.flatnonzero(c > t)
    if above.size:
        v = int(above[0])
        lo = c[v - 1] if v > 0 else 0
        margin = min(u - lo / total, c[v] / total - u)
        return v, margin
    positive = np.flatnonzero(np.asarray(weights) > 0)
    return int(positive[-1]), 0


# ---------------------------------------------------------------------------
# chain
# ---------------------------------------------------------------------------

def walk_chain(gamma, V, get_p, get_q, tokens, u_accept, u_draw):
    """Verify one draft chain.

    whoami-wesleyyou.top "Speculative Decoding" notes, § 从单个 token 接到一段
    draft: check positions in order; at the first rejected position j sample
    the correction from norm([p_j - q_j]_+) and drop the rest; if all gamma
    drafts are accepted, sample a bonus token from p_{gamma+1}.
    tannlonggtaoo.github.io "Speculative Decoding", § 算法 (the same loop with
    the bonus token at the last position) and § Greedy Sampling (temperature
    0: accept iff the draft equals the argmax; the correction is the argmax).

    get_p(i) -> Dist for target position i (0..gamma), get_q(i) -> Dist for
    draft position i (0..gamma-1); u_accept(i), u_draw(i) -> uniforms.
    A one-hot target row (greedy, or a non-finite row's fallback) takes the
    greedy rule and never reads q.

    Returns a dict: num_accepted, tokens (gamma+1, -1 padded), flags,
    final_dist (the distribution the last token was drawn from, None for a
    bonus draw), decisions [(i, |u - alpha|)], draw_margin, j.
    """
    flags = 0
    out = []
    decisions = []
    for i in range(gamma + 1):
        p = get_p(i)
        flags |= p.flags
        if i == gamma:
            if p.onehot:
                token, margin = p.index, None
            else:
                token, margin = inverse_cdf(p.probs, u_draw(i))
            return _chain_result(gamma, out, token, flags, None, decisions, margin)
        x = int(tokens[i])
        if p.onehot:
            if not (0 <= x < V):
                flags |= FLAG_BAD_TOKEN
            if x == p.index:
                out.append(x)
                continue
            return _chain_result(gamma, out, p.index, flags, p.dense(V), decisions, None)
        q = get_q(i)
        flags |= q.flags
        qv = q.dense(V, dtype=np.asarray(p.probs).dtype)
        u = u_accept(i)
        accepted, alpha, f = accept_test(p.probs, qv, x, u)
        flags |= f
        if f == 0:
            decisions.append((i, abs(u - alpha)))
        if accepted:
            out.append(x)
            continue
        r, _, f = positive_residual(p.probs, qv)
        if f:
            flags |= f
            r = p.probs
        token, margin = inverse_cdf(r, u_draw(i))
        return _chain_result(gamma, out, token, flags, r, decisions, margin)
    raise AssertionError("unreachable")


def _chain_result(gamma, accepted, token, flags, final_dist, decisions, margin):
    toks = list(accepted) + [token]
    toks += [-1] * (gamma + 1 - len(toks))
    return dict(num_accepted=len(accepted), tokens=toks, flags=flags,
                final_dist=final_dist, decisions=decisions, draw_margin=margin,
                j=len(accepted))


def chain_uniforms(seed, seq, uniform_override):
    """(u_accept, u_draw) callables for sequence ``seq`` of a chain batch."""
    if uniform_override is not None:
        ov = np.asarray(uniform_override, dtype=np.float64)
        return (lambda i: float(ov[seq, i, 0])), (lambda i: float(ov[seq, i, 1]))
    return ((lambda i: philox.uniform(seed, seq, i, 0)),
            (lambda i: philox.uniform(seed, seq, i, 1)))


def _per_seq(x, n, default):
    return np.full(n, default, np.float64) if x is None else np.asarray(x, np.float64)


def verify_chain(target_logits, draft_logits, draft_tokens, target_temperature,
                 draft_temperature, target_top_k=None, draft_top_k=None,
                 seed=0, uniform_override=None, seqs=None, target_top_p=None,
                 draft_top_p=None, target_min_p=None, draft_min_p=None):
    """Logit-level chain verification for a batch.

    target_logits [B, gamma+1, V], draft_logits [B, gamma, V] (any real
    dtype, converted exactly to float64 row by row), draft_tokens [B, gamma],
    per-sequence temperatures and top-k, and optionally per-sequence top-p and
    min-p (oracle.policy.policy_distribution_ext; None: no filter).  Rows are
    processed lazily: only the rows up to the first rejection are touched,
    like the pages' loop.
    Returns a list of per-sequence dicts (see ``walk_chain``).
    """
    B, G1, V = target_logits.shape
    gamma = G1 - 1
    kp = np.zeros(B, np.int64) if target_top_k is None else np.asarray(target_top_k)
    kq = np.zeros(B, np.int64) if draft_top_k is None else np.asarray(draft_top_k)
    pp, pq = _per_seq(target_top_p, B, 1.0), _per_seq(draft_top_p, B, 1.0)
    mp, mq = _per_seq(target_min_p, B, 0.0), _per_seq(draft_min_p, B, 0.0)
    results = []
    for b in (range(B) if seqs is None else seqs):
        def get_p(i, b=b):
            return policy_distribution_ext(np.asarray(target_logits[b, i], np.float64),
                                           target_temperature[b], kp[b], pp[b], mp[b])

        def get_q(i, b=b):
            return policy_distribution_ext(np.asarray(draft_logits[b, i], np.float64),
                                           draft_temperature[b], kq[b], pq[b], mq[b])

        ua, ud = chain_uniforms(seed, b, uniform_override)
        res = walk_chain(gamma, V, get_p, get_q, draft_tokens[b], ua, ud)
        res["seq"] = b
        results.append(res)
    return results


# ---------------------------------------------------------------------------
# tree
# ---------------------------------------------------------------------------

def overlap(p, q):
    """beta = sum_x min(p(x), q(x)): the acceptance rate of one position.

    whoami-wesleyyou.top "Speculative Decoding" notes, § Correction 为什么用正
    残差 (beta := sum_x min{p(x), q(x)}, Z := 1 - beta = sum_x [p(x) - q(x)]_+;
    beta = 1 when p = q) and § 手稿中的数值例子 (beta = 0.7).

    Works on float64 and on Fraction arrays.  Parity: pinned (the page's
    worked examples, the identity beta + Z = 1 against positive_residual,
    p = q, disjoint supports).
    """
    return np.minimum(p, q).sum()


def chain_overlap(target_logits, draft_logits, target_temperature, draft_temperature,
                  target_top_k=None, draft_top_k=None):
    """beta_i for every draft position i of every sequence: [B, gamma] float64.

    Each side's policy is applied as in verify_chain (oracle.policy), then
    overlap(p_i, q_i).  Rows whose policy flags them non-finite use their
    one-hot fallback, as the verifier does.
    """
    B, G1, V = target_logits.shape
    gamma = G1 - 1
    out = np.zeros((B, gamma))
    for b in range(B):
        kp = 0 if target_top_k is None else int(target_top_k[b])
        kq = 0 if draft_top_k is None else int(draft_top_k[b])
        for i in range(gamma):
            p = policy_distribution(target_logits[b, i], float(target_temperature[b]), kp).dense(V)
            q = policy_distribution(draft_logits[b, i], float(draft_temperature[b]), kq).dense(V)
            out[b, i] = overlap(p, q)
    return out


# ---------------------------------------------------------------------------
# typical acceptance (approximate, not distribution-exact)
# ---------------------------------------------------------------------------

def entropy(p):
    """H(p) = -sum_x p(x) ln p(x), natural log, with 0 ln 0 = 0."""
    p = np.asarray(p, dtype=np.float64)
    nz = p > 0
    return float(-(p[nz] * np.log(p[nz])).sum())


def typical_threshold(p, epsilon, delta):
    """min(epsilon, delta * exp(-H(p))): the probability a draft token must exceed.

    whoami-wesleyyou.top "Speculative Decoding" notes, § Medusa-1 与 typical
    acceptance (the criterion p(x_i | x_<i) > min{epsilon, delta
    exp[-H(p(. | x_<i))]}, H the entropy; epsilon a fixed threshold, delta
    scaling the entropy-dependent one).
    """
    return min(float(epsilon), float(delta) * float(np.exp(-entropy(p))))


def walk_typical(gamma, V, get_p, get_z, tokens, epsilon, delta):
    """Typical acceptance of one draft chain.

    whoami-wesleyyou.top "Speculative Decoding" notes, § Medusa-1 与 typical
    acceptance: each draft token x_i is tested against the target's own
    distribution at its position with p(x_i) > min(epsilon, delta exp(-H)),
    the longest prefix that passes is kept, and the token that follows it is
    the target's greedy choice, accepted without a test.  The rule trades the
    exactness of the min(1, p/q) test for speed: its output law is not the
    target's (also jennyma11.github.io "11.3 Self-Draft: Medusa、EAGLE-2/3 与
    Draft Tree", § 11.3.1: typical acceptance is an approximate acceptance
    mode).

    get_p(i) -> Dist of target position i after its policy; get_z(i) -> raw
    logits of that row (for the greedy token).  A draft token outside [0, V)
    fails its test and sets FLAG_BAD_TOKEN.  Returns a dict: num_accepted,
    tokens (gamma + 1, -1 padded), flags, decisions [(i, p(x_i), threshold)].
    """
    flags = 0
    out = []
    decisions = []
    for i in range(gamma + 1):
        p = get_p(i)
        flags |= p.flags
        if i < gamma:
            x = int(tokens[i])
            if 0 <= x < V:
                dense = p.dense(V)
                px = float(dense[x])
                thr = typical_threshold(dense, epsilon, delta)
                decisions.append((i, px, thr))
                if px > thr:
                    out.append(x)
                    continue
            else:
                flags |= FLAG_BAD_TOKEN
        greedy = p.index if p.onehot else finite_argmax(get_z(i))
        toks = out + [greedy]
        toks += [-1] * (gamma + 1 - len(toks))
        return dict(num_accepted=len(out), tokens=toks, flags=flags, decisions=decisions)
    raise AssertionError("unreachable")


def typical_chain(target_logits, draft_tokens, target_temperature, epsilon, delta, seqs=None):
    """Typical acceptance for a batch: target_logits [B, gamma+1, V], draft_tokens
    [B, gamma], a temperature per sequence (top-k is not part of this rule's
    interface).  Rows are read lazily, up to the first failed test."""
    B, G1, V = target_logits.shape
    gamma = G1 - 1
    results = []
    for b in (range(B) if seqs is None else seqs):
        def get_z(i, b=b):
            return np.asarray(target_logits[b, i], np.float64)

        def get_p(i, b=b):
            return policy_distribution(get_z(i), target_temperature[b], 0)

        res = walk_typical(gamma, V, get_p, get_z, draft_tokens[b], epsilon, delta)
        res["seq"] = b
        results.append(res)
    return results


def tree_check(parent, max_depth):
    """Validate a parent array; returns (flags, depth list or None).

    Node 0 is the root (parent -1); every other node n needs 0 <= parent[n] < n
    (breadth-first style numbering, as the pages' flattened trees).  A tree
    deeper than max_depth is flagged FLAG_DEPTH.
    """
    N = len(parent)
    if N == 0 or int(parent[0]) != -1:
        return FLAG_BAD_TREE, None
    depth = [0] * N
    for n in range(1, N):
        a = int(parent[n])
        if not (0 <= a < n):
            return FLAG_BAD_TREE, None
        depth[n] = depth[a] + 1
    if max(depth) > max_depth:
        return FLAG_DEPTH, depth
    return 0, depth


def walk_tree(N, V, parent, tokens, get_p, get_q, u_accept, u_draw, max_depth):
    """Recursive rejection over a candidate tree.

    whoami-wesleyyou.top "Speculative Decoding" notes, § Token Tree Verifier
    (multi-step speculative sampling: after rejecting a candidate, update the
    residual and test the next candidate; siblings are not retried
    independently against the original p); zzszmyf.github.io
    "LLM 推测解码精读笔记 · 04 EAGLE：特征空间草稿", § 6.2 验证阶段 (accept t
    iff r <= min(1, p(t)/q(t)), otherwise resample from norm(max(0, p - q)),
    recursively node by node); jennyma11.github.io "11.3 Self-Draft", § 11.3.4
    Tree Attention.

    Reading (config text of the tree workload): children of a node are its
    nodes with parent == node, tested in ascending id; on acceptance move to
    the child with its own target row; on rejection p <- norm([p - q_node]_+)
    and try the next child; when every child is rejected draw from the
    current p; at a leaf draw the bonus from p_leaf.  A degenerate residual
    leaves p unchanged and is flagged.  An invalid or too deep tree gives no
    result (num_accepted = -1).

    get_p(n), get_q(n) -> Dist of node n's target / draft rows;
    u_accept(c) -> acceptance uniform of child c; u_draw(n) -> draw uniform
    at node n.
    """
    width = max_depth + 1
    tflags, _ = tree_check(parent, max_depth)
    if tflags:
        return dict(num_accepted=-1, path=[-1] * width, tokens=[-1] * width,
                    flags=tflags, final_dist=None, decisions=[], draw_margin=None)
    children = [[] for _ in range(N)]
    for c in range(1, N):
        children[int(parent[c])].append(c)
    cur = 0
    path = [0]
    out = []
    flags = 0
    decisions = []
    while True:
        p = get_p(cur)
        flags |= p.flags
        kids = children[cur]
        if p.onehot:
            nxt = None
            for c in kids:
                x = int(tokens[c])
                if not (0 <= x < V):
                    flags |= FLAG_BAD_TOKEN
                if x == p.index:
                    nxt = c
                    break
            if nxt is not None:
                cur = nxt
                path.append(cur)
                out.append(int(tokens[cur]))
                continue
            final = p.dense(V) if kids else None
            return _tree_result(width, path, out, p.index, flags, final, decisions, None)
        if not kids:
            token, margin = inverse_cdf(p.probs, u_draw(cur))
            return _tree_result(width, path, out, token, flags, None, decisions, margin)
        q = get_q(cur)
        flags |= q.flags
        qv = q.dense(V, dtype=np.asarray(p.probs).dtype)
        dist = p.probs
        nxt = None
        for c in kids:
            u = u_accept(c)
            accepted, alpha, f = accept_test(dist, qv, tokens[c], u)
            flags |= f
            if f == 0:
                decisions.append((c, abs(u - alpha)))
            if accepted:
                nxt = c
                break
            r, _, f = positive_residual(dist, qv)
            if f:
                flags |= f
            else:
                dist = r
        if nxt is not None:
            cur = nxt
            path.append(cur)
            out.append(int(tokens[cur]))
            continue
        token, margin = inverse_cdf(dist, u_draw(cur))
        return _tree_result(width, path, out, token, flags, dist, decisions, margin)


def _tree_result(width, path, accepted, token, flags, final_dist, decisions, margin):
    p = list(path) + [-1] * (width - len(path))
    t = list(accepted) + [token]
    t += [-1] * (width - len(t))
    return dict(num_accepted=len(accepted), path=p, tokens=t, flags=flags,
                final_dist=final_dist, decisions=decisions, draw_margin=margin)


def tree_uniforms(seed, tree, uniform_override):
    """(u_accept(child), u_draw(node)) callables for tree ``tree``."""
    if uniform_override is not None:
        ov = np.asarray(uniform_override, dtype=np.float64)
        return (lambda c: float(ov[tree, c, 0])), (lambda n: float(ov[tree, n, 1]))
    return ((lambda c: philox.uniform(seed, tree, c, 0)),
            (lambda n: philox.uniform(seed, tree, n, 1)))


def verify_tree(target_logits, draft_logits, node_tokens, parent, max_depth,
                target_temperature, draft_temperature, target_top_k=None,
                draft_top_k=None, seed=0, uniform_override=None, trees=None,
                target_top_p=None, draft_top_p=None, target_min_p=None, draft_min_p=None):
    """Logit-level tree verification for a batch of T trees of N nodes.

    target_logits [T, N, V]: row n is the target's next-token logits after the
    path root..n.  draft_logits [T, N, V]: row n is the draft logits that the
    children of n were drawn from.  node_tokens, parent [T, N].
    """
    T, N, V = target_logits.shape
    kp = np.zeros(T, np.int64) if target_top_k is None else np.asarray(target_top_k)
    kq = np.zeros(T, np.int64) if draft_top_k is None else np.asarray(draft_top_k)
    pp, pq = _per_seq(target_top_p, T, 1.0), _per_seq(draft_top_p, T, 1.0)
    mp, mq = _per_seq(target_min_p, T, 0.0), _per_seq(draft_min_p, T, 0.0)
    results = []
    for t in (range(T) if trees is None else trees):
        def get_p(n, t=t):
            return policy_distribution_ext(np.asarray(target_logits[t, n], np.float64),
                                           target_temperature[t], kp[t], pp[t], mp[t])

        def get_q(n, t=t):
            return policy_distribution_ext(np.asarray(draft_logits[t, n], np.float64),
                                           draft_temperature[t], kq[t], pq[t], mq[t])

        ua, ud = tree_uniforms(seed, t, uniform_override)
        res = walk_tree(N, V, parent[t], node_tokens[t], get_p, get_q, ua, ud, max_depth)
        res["tree"] = t
        results.append(res)
    return results


# ---------------------------------------------------------------------------
# tree mask and position ids
# ---------------------------------------------------------------------------

def tree_mask(parent, max_depth):
    """Ancestor-or-self mask and depth position ids for one tree.

    whoami-wesleyyou.top "Speculative Decoding" notes, § Token Tree Verifier:
    topology-aware causal mask (a node sees the shared prefix, its ancestors
    and itself, never another branch; positions follow path depth);
    jennyma11.github.io "11.3 Self-Draft", § 11.3.4 Tree Attention (position
    id by path depth, not by flattened index); wineandchord.com
    "推测解码：接受规则、状态与收益边界", § Tree Verification (parent, position
    and token arrays kept one-to-one).

    Returns (mask [N, ceil(N/64)] uint64, position [N] int32, flags).
    Bit m of mask[n] is set iff m == n or m is an ancestor of n.  Readings:
    position[n] is the depth when n's parent chain reaches the root through
    links with 0 <= parent[a] < a, else -1 (and the mask then holds the part
    of the chain that was reached); FLAG_BAD_TREE when parent[0] != -1 or any
    link is invalid; FLAG_DEPTH when a depth exceeds max_depth.
    """
    N = len(parent)
    words = (N + 63) // 64
    mask = np.zeros((N, words), dtype=np.uint64)
    position = np.full(N, -1, dtype=np.int32)
    flags = 0
    if N and int(parent[0]) != -1:
        flags |= FLAG_BAD_TREE
    for n in range(N):
        members = [n]
        a = n
        ok = True
        while a != 0:
            pa = int(parent[a])
            if not (0 <= pa < a):
                ok = False
                break
            members.append(pa)
            a = pa
        for m in members:
            mask[n, m // 64] |= np.uint64(1) << np.uint64(m % 64)
        if ok:
            position[n] = len(members) - 1
            if position[n] > max_depth:
                flags |= FLAG_DEPTH
        else:
            flags |= FLAG_BAD_TREE
    return mask, position, flags


# ---------------------------------------------------------------------------
# EAGLE-2 rerank of a draft tree
# ---------------------------------------------------------------------------

def _dyadic(x):
    """A finite float as an exact pair (num, exp) with x = num * 2**exp."""
    m, e = math.frexp(float(x))
    if m == 0:
        return 0, 0
    num, exp = int(m * (1 << 53)), e - 53
    while num and num % 2 == 0:
        num //= 2
        exp += 1
    return num, exp


def tree_values(parent, confidence):
    """value(t_n) = product of the confidences c_j on the path root..t_n, exactly.

    zzszmyf.github.io "LLM 推测解码精读笔记 · 04 EAGLE：特征空间草稿",
    § 10.3 扩展 + 重排 (value(t_i) = prod over Path(root, t_i) of c_j).  Each
    confidence is taken as the exact value of its float32, and the product is
    formed in exact integer arithmetic: value[n] = (num, exp) with
    value = num * 2**exp.  Nothing is rounded, so the ranking below is the
    one the page's definition gives.  parent must be valid (tree_check).
    """
    c = np.asarray(confidence, dtype=np.float32)
    value = []
    for n in range(len(parent)):
        num, exp = _dyadic(c[n])
        if n:
            pn, pe = value[int(parent[n])]
            num, exp = num * pn, exp + pe
        value.append((num, exp) if num else (0, 0))
    return value


def value_float(v):
    """The float64 nearest an exact (num, exp) value (0 when it underflows);
    Python's integer true division rounds correctly."""
    num, exp = v
    return num / (1 << -exp) if exp < 0 else float(num << exp)


def value_keys(value):
    """Integers that order the exact values like the values themselves: each
    value scaled to the smallest exponent present."""
    emin = min((e for n, e in value if n), default=0)
    return [n << (e - emin) if n else 0 for n, e in value]


def clamp_confidence(confidence):
    """Confidences clamped into [0, 1] (NaN -> 0) and whether any was changed.

    The pages' properties (value(child) <= value(parent), a connected top-m)
    need c in [0, 1]; this entry point's reading is to clamp and flag."""
    c = np.asarray(confidence, dtype=np.float32)
    out = np.where(c > 0, np.minimum(c, np.float32(1)), np.float32(0)).astype(np.float32)
    changed = bool(np.isnan(c).any() or (c < 0).any() or (c > 1).any())
    return out, changed


def tree_rerank(parent, confidence, m):
    """EAGLE-2 rerank: the top-m nodes of a draft tree by value.

    zzszmyf.github.io "LLM 推测解码精读笔记 · 04 EAGLE：特征空间草稿",
    § 10.3 扩展 + 重排 (rerank: the m nodes of highest value over the whole
    tree, flattened into one sequence for verification; ties go to the
    shallower node; because c <= 1 a child's value never exceeds its parent's,
    so the chosen set is a connected tree) and § 题 5.  Reading: remaining
    ties go to the lower node index.  The ranking uses the exact path
    products of tree_values.

    Returns (nodes, new_parent, values, flags): the chosen node ids in
    ascending order (so parents precede children), each one's parent as a
    position in that list (-1 for the root), their values (the float64
    nearest each exact product), and flags (FLAG_BAD_TREE for an invalid
    parent array: nothing chosen; FLAG_NONFINITE when a confidence was
    clamped into [0, 1]).
    """
    N = len(parent)
    flags, depth = tree_check(parent, N)
    if flags & FLAG_BAD_TREE:
        return [], [], [], FLAG_BAD_TREE
    c, changed = clamp_confidence(confidence)
    flags = FLAG_NONFINITE if changed else 0
    value = tree_values(parent, c)
    key = value_keys(value)
    order = sorted(range(N), key=lambda n: (-key[n], depth[n], n))
    chosen = sorted(order[:min(m, N)])
    pos = {n: i for i, n in enumerate(chosen)}
    new_parent = [-1 if n == 0 else pos[int(parent[n])] for n in chosen]
    return chosen, new_parent, [value_float(value[n]) for n in chosen], flags


def rerank_order(parent, confidence):
    """Every node of a valid tree in rerank order (best first) with its exact
    value and depth: the ranking tree_rerank cuts at m."""
    N = len(parent)
    _, depth = tree_check(parent, N)
    c, _ = clamp_confidence(confidence)
    value = tree_values(parent, c)
    key = value_keys(value)
    order = sorted(range(N), key=lambda n: (-key[n], depth[n], n))
    return order, value, depth
