"""Float64 restatement of DFlash drafting at temperature > 0 (oracle; test
infrastructure).

Only tests, the smoke entry and the bench's CPU-baseline leg may import this.

The pages report DFlash with sampling (temperature = 1) beside greedy
decoding ([Paper walkthrough] Results; [News summary] 用例与示例, reasoning
models) and describe one verification step for both: the drafter's block is
compared position by position with the target model's sampled tokens and the
longest matching prefix (cumulative product of the matches) is kept, the
target's own token at the first mismatch being the bonus ([Code walkthrough]
§三 第3步).  So at temperature T > 0 only the token choice changes, on both
sides: each block row i = 1..S-1 draws its draft from its own
q_i = softmax(z_i / T) (z: the drafter's logits), and the verifier draws its
tokens from its own distribution; acceptance is the same longest-prefix rule
as greedy decoding (dflash_ref.accept_longest_prefix).  T -> 0 recovers the
greedy argmax.

A draw from softmax(z / T) is made by the Gumbel-max rule:
argmax_v (z(v)/T + g(v)) with independent standard Gumbel g.  The random
numbers come from one counter-based generator, SplitMix64 (Steele, Lea and
Flood, OOPSLA 2014): a stream key folds (seed, purpose, request, round,
row), and element v of the stream is mix(key + (v+1) * golden).  The CUDA
path implements the same published function on its own.  Uniforms use the
top 23 bits, u = ((bits >> 41) + 1/2) * 2^-23, so each lies strictly inside
(0, 1) and is exact in float32; g = -ln(-ln u).
"""
from __future__ import annotations

import numpy as np

DRAFT = 1   # purpose id of the drafter's Gumbel streams
TARGET = 2  # purpose id of the target's Gumbel streams

_MASK = (1 << 64) - 1
_GOLD = 0x9E3779B97F4A7C15


def _mix(z):
    """SplitMix64 output mix (the published two-multiply finaliser), on a
    Python int or a uint64 array."""
    if isinstance(z, np.ndarray):
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        return z ^ (z >> np.uint64(31))
    z &= _MASK
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK
    return z ^ (z >> 31)


def stream_key(seed: int, *ids: int) -> int:
    """Fold a seed and integer ids into one 64-bit stream key."""
    k = _mix((int(seed) + _GOLD) & _MASK)
    for i in ids:
        k = _mix((k + _GOLD * (int(i) + 1)) & _MASK)
    return k


def stream_bits(key: int, idx) -> np.ndarray:
    """Element idx of the stream started at key: mix(key + (idx+1) * golden)."""
    idx = np.asarray(idx, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(np.uint64(key) + (idx + np.uint64(1)) * np.uint64(_GOLD))


def uniform23(key: int, idx) -> np.ndarray:
    """Uniform in (0, 1): ((bits >> 41) + 1/2) * 2^-23."""
    b = stream_bits(key, idx) >> np.uint64(41)
    return (b.astype(np.float64) + 0.5) * 2.0 ** -23


def gumbel(key: int, idx) -> np.ndarray:
    """Standard Gumbel variates -ln(-ln u)."""
    return -np.log(-np.log(uniform23(key, idx)))


def sample_row(z: np.ndarray, temperature: float, key: int) -> tuple[int, float]:
    """One draw from softmax(z / T) by the Gumbel-max rule, ties to the lowest
    id; returns the index and the top-1 minus top-2 margin of the perturbed
    scores (how far the draw is from flipping)."""
    pert = z / temperature + gumbel(key, np.arange(z.shape[-1]))
    i = int(np.argmax(pert))
    top2 = np.partition(pert, -2)[-2:]
    return i, float(top2[1] - top2[0])


def sample_drafts(z: np.ndarray, temperature: float, seed: int, b: int, rnd: int):
    """Drafts of block rows 1..S-1 of request b in round rnd from their logits
    z [S-1, V] (row k holds block row k+1), each drawn from softmax(z_i / T)
    with the stream (seed, DRAFT, b, rnd, i).  Returns (drafts, margins)."""
    d, mg = [], []
    for k in range(z.shape[0]):
        idx, m = sample_row(z[k], temperature, stream_key(seed, DRAFT, b, rnd, k + 1))
        d.append(idx)
        mg.append(m)
    return np.array(d, dtype=np.int64), np.array(mg)


def sample_target_rows(z: np.ndarray, temperature: float, seed: int, slot: int, pos0: int):
    """The target's sampled tokens for block rows at positions pos0, pos0+1, ..
    of request `slot` (the verify step at temperature T > 0): row i's token
    -- the one that follows position pos0+i -- is drawn from softmax(z_i / T)
    with the stream (seed, TARGET, slot, pos0+i).  Keyed by position, not by
    round, so the speculative loop and the target's own sampled decoding draw
    the same numbers for the same position.  Returns (tokens, margins)."""
    d, mg = [], []
    for i in range(z.shape[0]):
        idx, m = sample_row(z[i], temperature, stream_key(seed, TARGET, slot, pos0 + i))
        d.append(idx)
        mg.append(m)
    return np.array(d, dtype=np.int64), np.array(mg)
