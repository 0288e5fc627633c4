"""Philox4x32-10 counter-based generator, written from its published definition.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Source: J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel random
numbers: as easy as 1, 2, 3", SC'11, section on the Philox family: a 4x32
block of counter words is transformed by R rounds; each round multiplies
words 0 and 2 by two fixed odd constants, keeps the high and low halves of
the 64-bit products, and mixes the high halves with words 1 and 3 and the
two key words; the key is advanced by two Weyl constants between rounds.

Why a counter-based generator: the pages ask that a fixed seed replay the
same run and warn that different acceptance paths otherwise consume the
generator a different number of times (wineandchord.com
"推测解码：接受规则、状态与收益边界", § 常见失效 "固定 seed 不可重放" and
§ 状态事务 "advance stream and RNG exactly once").  Keying every draw by
(seed, sequence, position, draw) makes each uniform independent of the path.

Keying used by the verifier (a reading of ours; the pages name no generator,
so this layout is "parity unpinned by the pages" and is pinned only by the
published known-answer vectors of Philox4x32-10 and by oracle<->GPU parity):
  key     = (seed & 0xffffffff, seed >> 32)
  counter = (seq, pos, draw, 0)
  draw 0  = acceptance uniform, draw 1 = inverse-CDF (correction/bonus) uniform
  u       = (word0 >> 8) * 2**-24, so u lies in [0, 1) on a 2**-24 grid.
"""

MASK32 = 0xFFFFFFFF

# Round multipliers and key increments of Philox4x32 (SC'11 paper).
PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85


def philox4x32(counter, key, rounds=10):
    """Return the four 32-bit output words for a 4-word counter and 2-word key."""
    x0, x1, x2, x3 = (int(c) & MASK32 for c in counter)
    k0, k1 = (int(k) & MASK32 for k in key)
    for _ in range(rounds):
        prod0 = PHILOX_M0 * x0
        prod1 = PHILOX_M1 * x2
        hi0, lo0 = prod0 >> 32, prod0 & MASK32
        hi1, lo1 = prod1 >> 32, prod1 & MASK32
        x0, x1, x2, x3 = hi1 ^ x1 ^ k0, lo1, hi0 ^ x3 ^ k1, lo0
        k0 = (k0 + PHILOX_W0) & MASK32
        k1 = (k1 + PHILOX_W1) & MASK32
    return x0, x1, x2, x3


def uniform(seed, seq, pos, draw):
    """Uniform in [0, 1) for one (seed, seq, pos, draw) key, as a Python float."""
    seed = int(seed)
    key = (seed & MASK32, (seed >> 32) & MASK32)
    w0 = philox4x32((seq, pos, draw, 0), key)[0]
    return (w0 >> 8) * (2.0 ** -24)
