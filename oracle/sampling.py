"""Target-only sampled verification: random numbers and the sampled pick (TEST
INFRASTRUCTURE ONLY).

[DMTP] "DMTP: A Better First Token for Block Drafting via MTP", §5: the experiments
verify against the target alone, comparing each candidate in turn with the token the
target samples there and keeping the matched prefix; §7 runs every method at temperature
1. [colibri] verify contract: every pick, whether greedy or sampled, comes from the
target's own full logits and the sampler never sees the drafts; a draft counts as
accepted exactly when the target's sample equals it.

Reading (the pages name no sampler or generator): the target's token at position p of
sequence b is the Gumbel-max sample argmax_v (l_v / temperature + G_v) of its logits
l, which is an exact draw from softmax(l / temperature); G_v = -log(-log u_v), and u_v
comes from the counter-based generator Philox4x32-10 (Salmon, Moraes, Dror and Shaw,
"Parallel random numbers: as easy as 1, 2, 3", SC 2011) keyed by the sampling seed and
counted by (v / 4, p, b, 0), word v mod 4, u = (word >> 8 + 1/2) 2^-24. Keying the noise
by position (not by round) makes speculative output equal plain sampled decoding with
the same noise. The drafts (T1 from MTP, T2..T7 from the drafter) stay argmax picks.
"""
from __future__ import annotations

import numpy as np

_M0, _M1 = 0xD2511F53, 0xCD9E8D57   # Philox4x32 round multipliers
_W0, _W1 = 0x9E3779B9, 0xBB67AE85   # Weyl key increments
_MASK = 0xFFFFFFFF


def philox4x32_10(ctr, key):
    """Philox4x32 with 10 rounds on arrays: ctr (4, n) and key (2,) or (2, n) of uint32
    values; returns (4, n) uint32. Each round multiplies words 0 and 2 by the round
    constants, and the new words are (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1,
    lo(M0 c0)); the key takes a Weyl step between rounds."""
    c = [np.asarray(x, dtype=np.uint64) & _MASK for x in ctr]
    k0 = np.asarray(key[0], dtype=np.uint64) & _MASK
    k1 = np.asarray(key[1], dtype=np.uint64) & _MASK
    for r in range(10):
        p0 = c[0] * np.uint64(_M0)
        p1 = c[2] * np.uint64(_M1)
        hi0, lo0 = p0 >> np.uint64(32), p0 & np.uint64(_MASK)
        hi1, lo1 = p1 >> np.uint64(32), p1 & np.uint64(_MASK)
        c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
        if r < 9:
            k0 = (k0 + np.uint64(_W0)) & np.uint64(_MASK)
            k1 = (k1 + np.uint64(_W1)) & np.uint64(_MASK)
    return np.stack([x.astype(np.uint32) for x in c])


def seed_key(seed: int):
    return np.array([seed & _MASK, (seed >> 32) & _MASK], dtype=np.uint64)


def uniforms(seed: int, b: int, pos: int, vocab: int) -> np.ndarray:
    """u_v for v = 0..vocab-1 at (sequence b, position pos), float64 in (0, 1)."""
    nblk = (vocab + 3) // 4
    ctr = np.zeros((4, nblk), dtype=np.uint64)
    ctr[0] = np.arange(nblk, dtype=np.uint64)
    ctr[1] = pos
    ctr[2] = b
    w = philox4x32_10(ctr, seed_key(seed))          # (4, nblk): word i of block j is v = 4j + i
    words = w.T.reshape(-1)[:vocab]
    return ((words >> np.uint32(8)).astype(np.float64) + 0.5) * 2.0 ** -24


def gumbel(seed: int, b: int, pos: int, vocab: int) -> np.ndarray:
    u = uniforms(seed, b, pos, vocab)
    return -np.log(-np.log(u))


def sampled_scores(logits, temperature: float, seed: int, b: int, pos: int) -> np.ndarray:
    """l / temperature + G: their argmax is the target's sample at (b, pos)."""
    logits = np.asarray(logits, dtype=np.float64)
    return logits / temperature + gumbel(seed, b, pos, logits.shape[-1])
