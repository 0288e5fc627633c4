"""Seeded synthetic verification workloads.

This module only builds inputs: logits, draft tokens, trees and policies.  It
holds none of the verifier's arithmetic (no softmax, no acceptance ratio, no
residual): draft tokens are drawn with the Gumbel-max trick,
argmax_v(z_v / T + G_v) with G_v = -log(-log U_v), which samples from
softmax(z / T) without forming it.  Both the CUDA path's tests and the CPU
oracle read the arrays made here.

Recipe (all numpy PCG64, generator seed given per workload):
  z_p[row, v] = scale * N(0, 1) - zipf * log(rank[v] + 1)
      rank = one seeded permutation of the vocabulary per workload (token v has
      Zipf rank rank[v]; the same ranks for every row);
  z_q = z_p + N(0, sigma^2) drawn independently per element;
  both rounded to bf16 (round to nearest even) for bf16 workloads, kept as
  float32 otherwise; values are returned as float32 arrays holding exactly
  the stored values;
  draft tokens are drawn from the draft's own policy on the stored values:
  softmax(z_q / T) (Gumbel-max), top-k (Gumbel-max over the k largest), or
  the argmax for temperature 0.

Workloads 0-4 are the five configurations the library is measured on:
  0  chain  B=4   gamma=4 V=32000  fp32 scale 2   zipf 1.1 sigma 0.5 T=1
  1  chain  B=64  gamma=5 V=32000  bf16 scale 2   zipf 1.1 sigma 0.7 T=0.8
  2  chain  B=256 gamma=7 V=128256 bf16 scale 2.5 zipf 1.2 sigma 0.4 T=1
  3  chain  B=128 gamma=4 V=152064 bf16 scale 2.5 zipf 1.2 sigma 0.5;
            sequences 0-63 greedy (T=0 both sides, draft = argmax q),
            sequences 64-127 top-k 50 at T=0.7 on both sides
  4  tree   32 trees x 60 nodes, V=128256 bf16, scale 2.5 zipf 1.2 sigma 0.5,
            T=1; a full tree with branching 4,3,2,2,1,1 by depth (185 nodes)
            pruned by removing uniformly chosen non-root leaves to 60 nodes,
            numbered breadth-first; children drawn i.i.d. from the parent's q.
"""

import numpy as np

PHILOX_SEED = 1234

CONFIGS = {
    0: dict(kind="chain", B=4, gamma=4, V=32000, dtype="f32", scale=2.0, zipf=1.1,
            sigma=0.5, temperature=1.0),
    1: dict(kind="chain", B=64, gamma=5, V=32000, dtype="bf16", scale=2.0, zipf=1.1,
            sigma=0.7, temperature=0.8),
    2: dict(kind="chain", B=256, gamma=7, V=128256, dtype="bf16", scale=2.5, zipf=1.2,
            sigma=0.4, temperature=1.0),
    3: dict(kind="chain", B=128, gamma=4, V=152064, dtype="bf16", scale=2.5, zipf=1.2,
            sigma=0.5, temperature=0.7, greedy_seqs=64, top_k=50),
    4: dict(kind="tree", T=32, N=60, V=128256, dtype="bf16", scale=2.5, zipf=1.2,
            sigma=0.5, temperature=1.0, branching=(4, 3, 2, 2, 1, 1)),
}


def round_bf16_inplace(x):
    """Round a float32 array to the nearest bf16 value (ties to even), in place."""
    bits = x.view(np.uint32)
    lsb = (bits >> np.uint32(16)) & np.uint32(1)
    bits += np.uint32(0x7FFF)
    bits += lsb
    bits &= np.uint32(0xFFFF0000)
    return x


def _logits(rng, shape, V, scale, zipf, dtype, perm_rng=None):
    """scale * N(0,1) - zipf * log(rank + 1), float32 (bf16-rounded if asked)."""
    ranks = (perm_rng or rng).permutation(V)
    bias = (-zipf * np.log(ranks.astype(np.float64) + 1.0)).astype(np.float32)
    z = rng.standard_normal(size=shape + (V,), dtype=np.float32)
    z *= np.float32(scale)
    z += bias
    return z, bias


def _noisy_copy(rng, z, sigma):
    out = rng.standard_normal(size=z.shape, dtype=np.float32)
    out *= np.float32(sigma)
    out += z
    return out


def gumbel_argmax(rng, z_row, temperature, top_k=0):
    """One draw from the draft policy of a row, by Gumbel-max (T=0: argmax)."""
    z_row = np.asarray(z_row, dtype=np.float64)
    if temperature == 0:
        return int(np.argmax(z_row))
    idx = np.arange(z_row.shape[0])
    if 0 < top_k < z_row.shape[0]:
        idx = np.argpartition(-z_row, top_k - 1)[:top_k]
    u = rng.random(idx.shape[0])
    u = np.clip(u, 1e-300, 1.0 - 1e-16)
    g = -np.log(-np.log(u))
    return int(idx[np.argmax(z_row[idx] / temperature + g)])


def make_chain(B, gamma, V, dtype="bf16", scale=2.5, zipf=1.2, sigma=0.4,
               temperature=1.0, seed=0, greedy_seqs=0, top_k=0):
    """A chain batch: target [B, gamma+1, V], draft [B, gamma, V], tokens [B, gamma].

    Sequences < greedy_seqs use temperature 0 on both sides (draft token =
    argmax of the draft row); the others use ``temperature`` and ``top_k``.
    """
    rng = np.random.default_rng(seed)
    target, _ = _logits(rng, (B, gamma + 1), V, scale, zipf, dtype)
    draft = _noisy_copy(rng, target[:, :gamma], sigma)
    if dtype == "bf16":
        round_bf16_inplace(target)
        round_bf16_inplace(draft)
    temps = np.full(B, temperature, dtype=np.float32)
    topk = np.full(B, top_k, dtype=np.int32)
    temps[:greedy_seqs] = 0.0
    topk[:greedy_seqs] = 0
    tokens = np.zeros((B, gamma), dtype=np.int32)
    trng = np.random.default_rng(seed + 7_000_003)
    for b in range(B):
        for i in range(gamma):
            tokens[b, i] = gumbel_argmax(trng, draft[b, i], float(temps[b]), int(topk[b]))
    return dict(kind="chain", B=B, gamma=gamma, V=V, dtype=dtype,
                target=target, draft=draft, tokens=tokens,
                target_temperature=temps.copy(), draft_temperature=temps.copy(),
                target_top_k=topk.copy(), draft_top_k=topk.copy(),
                seed=PHILOX_SEED)


def tree_shape(rng, branching, n_nodes):
    """Parent array of a pruned full tree, numbered breadth-first (parent < id)."""
    parents = [-1]
    depth = [0]
    frontier = [0]
    for b in branching:
        nxt = []
        for node in frontier:
            for _ in range(b):
                parents.append(node)
                depth.append(depth[node] + 1)
                nxt.append(len(parents) - 1)
        frontier = nxt
    alive = set(range(len(parents)))
    n_children = [0] * len(parents)
    for n in range(1, len(parents)):
        n_children[parents[n]] += 1
    while len(alive) > n_nodes:
        leaves = sorted(n for n in alive if n != 0 and n_children[n] == 0)
        victim = leaves[int(rng.integers(len(leaves)))]
        alive.remove(victim)
        n_children[parents[victim]] -= 1
    order = sorted(alive)
    new_id = {old: i for i, old in enumerate(order)}
    return np.array([-1] + [new_id[parents[old]] for old in order[1:]], dtype=np.int32)


def make_tree(T, N, V, dtype="bf16", scale=2.5, zipf=1.2, sigma=0.5, temperature=1.0,
              branching=(4, 3, 2, 2, 1, 1), seed=0, parents=None, top_k=0):
    """A tree batch: target/draft [T, N, V], node_tokens and parent [T, N]."""
    rng = np.random.default_rng(seed)
    target, _ = _logits(rng, (T, N), V, scale, zipf, dtype)
    draft = _noisy_copy(rng, target, sigma)
    if dtype == "bf16":
        round_bf16_inplace(target)
        round_bf16_inplace(draft)
    srng = np.random.default_rng(seed + 5_000_011)
    if parents is None:
        parent = np.stack([tree_shape(srng, branching, N) for _ in range(T)])
    else:
        parent = np.broadcast_to(np.asarray(parents, np.int32), (T, N)).copy()
    temps = np.full(T, temperature, dtype=np.float32)
    topk = np.full(T, top_k, dtype=np.int32)
    tokens = np.zeros((T, N), dtype=np.int32)
    trng = np.random.default_rng(seed + 7_000_003)
    for t in range(T):
        for n in range(1, N):
            tokens[t, n] = gumbel_argmax(trng, draft[t, parent[t, n]], float(temps[t]),
                                         int(topk[t]))
    return dict(kind="tree", T=T, N=N, V=V, dtype=dtype, target=target, draft=draft,
                tokens=tokens, parent=parent, max_depth=len(branching),
                target_temperature=temps.copy(), draft_temperature=temps.copy(),
                target_top_k=topk.copy(), draft_top_k=topk.copy(), seed=PHILOX_SEED)


def make_rerank(T, N, seed=0, width=8, levels=256, deep=False):
    """Draft trees for the rerank: parent [T, N] int32 and confidence [T, N]
    float32.

    Node n > 0 hangs under a node drawn uniformly from the previous `width`
    ids (bushy trees a few levels deep; deep=True: a single chain).
    Confidences are a draft's top probabilities, Beta(2, 1)-shaped, on a grid
    of `levels` steps so that equal values (and equal path products) occur;
    the root's is 1.
    """
    rng = np.random.default_rng(seed)
    parent = np.empty((T, N), np.int32)
    parent[:, 0] = -1
    for n in range(1, N):
        parent[:, n] = n - 1 if deep else rng.integers(max(0, n - width), n, size=T)
    conf = np.sqrt(rng.random((T, N)))
    conf = (np.ceil(conf * levels) / levels).astype(np.float32)
    conf[:, 0] = 1.0
    return dict(parent=parent, confidence=conf)


def config(i):
    """Inputs of workload i (0-4), generator seed 1000 + i."""
    c = dict(CONFIGS[i])
    kind = c.pop("kind")
    if kind == "chain":
        return make_chain(seed=1000 + i, **c)
    return make_tree(seed=1000 + i, **c)
