"""Counter-based random streams of the gating variants, float64 / exact
integer reference.

TEST INFRASTRUCTURE ONLY (see ``moe_oracle``): imported by the oracle, the
tests and the bench's oracle legs; the product path never imports it.  It
shares no code with the CUDA library, which implements the same generator
from the same published definition.

The deepspeed.moe overview (adg.csdn.net/694deb285b9f5f31781ae763, §2.1)
names three randomised gate options without giving formulas:
``noisy_gate_policy`` (jitter or rsample, against expert-selection bias),
``use_rts`` (random token selection) and ``top2_2nd_expert_sampling``.  The
layer draws their randomness itself, so that a run is reproducible from a
seed and an offset (readings R11-R14 of the oracle module):

* Generator: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random
  numbers: as easy as 1, 2, 3", SC 2011): 10 rounds on a 4 x 32-bit counter
  with a 2 x 32-bit key, multipliers 0xD2511F53 / 0xCD9E8D57, key increments
  0x9E3779B9 / 0xBB67AE85.  Key = (seed low word, seed high word).
* Streams: counter = (index, purpose << 24 | sub, offset low, offset high);
  purpose 1: the gate noise u[s, e] (index s, sub e // 4, word e % 4);
  purpose 2: the jitter u[s, c] (index s, sub c // 4, word c % 4);
  purpose 3: round r of the RTS permutation's Feistel function (index = the
  round's input, sub = r, word 0).
* A 32-bit word w becomes u = ((w >> 9) + 0.5) * 2^-23, strictly inside
  (0, 1) and exactly representable in float32.
"""
from __future__ import annotations

import numpy as np

PHILOX_M0, PHILOX_M1 = 0xD2511F53, 0xCD9E8D57
PHILOX_W0, PHILOX_W1 = 0x9E3779B9, 0xBB67AE85
_MASK32 = np.uint64(0xFFFFFFFF)

PURPOSE_GATE_NOISE = 1
PURPOSE_JITTER = 2
PURPOSE_RTS = 3


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Philox4x32-10 on arrays of counters (broadcast); returns the four
    output words as uint64 arrays holding 32-bit values.

    Round: (c0, c1, c2, c3) <- (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2),
                                hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)),
    then the key advances by the Weyl increments."""
    c = [np.asarray(v, dtype=np.uint64) & _MASK32 for v in (c0, c1, c2, c3)]
    c = list(np.broadcast_arrays(*c))
    k0 = np.uint64(int(k0) & 0xFFFFFFFF)
    k1 = np.uint64(int(k1) & 0xFFFFFFFF)
    m0, m1 = np.uint64(PHILOX_M0), np.uint64(PHILOX_M1)
    for _ in range(10):
        p0 = m0 * c[0]          # < 2^64: no wrap
        p1 = m1 * c[2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK32
        c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
        k0 = np.uint64((int(k0) + PHILOX_W0) & 0xFFFFFFFF)
        k1 = np.uint64((int(k1) + PHILOX_W1) & 0xFFFFFFFF)
    return c


def uniform_open(words) -> np.ndarray:
    """u = ((w >> 9) + 0.5) * 2^-23 for 32-bit words w: the 23 high bits of
    the word, centred in their interval (float64, exact in float32 too)."""
    w = np.asarray(words, dtype=np.uint64) >> np.uint64(9)
    return (w.astype(np.float64) + 0.5) * 2.0 ** -23


def _key(seed):
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    return seed & 0xFFFFFFFF, seed >> 32


def stream_uniforms(num_rows: int, width: int, purpose: int, seed: int, offset: int) -> np.ndarray:
    """u[s, i] for s < num_rows, i < width of a purpose's stream (float64)."""
    k0, k1 = _key(seed)
    off = int(offset) & 0xFFFFFFFFFFFFFFFF
    s = np.arange(num_rows, dtype=np.uint64)[:, None]
    blocks = (width + 3) // 4
    sub = np.arange(blocks, dtype=np.uint64)[None, :] | np.uint64(purpose << 24)
    words = philox4x32_10(s, sub, off & 0xFFFFFFFF, off >> 32, k0, k1)
    full = np.stack(words, axis=-1).reshape(num_rows, blocks * 4)[:, :width]
    return uniform_open(full)


def gumbel(u) -> np.ndarray:
    """Standard Gumbel variates -ln(-ln u) (float64)."""
    u = np.asarray(u, dtype=np.float64)
    return -np.log(-np.log(u))


def gate_noise(num_tokens: int, num_experts: int, seed: int, offset: int):
    """(u, g): the gate's uniforms and their Gumbel variates, [S, E]."""
    u = stream_uniforms(num_tokens, num_experts, PURPOSE_GATE_NOISE, seed, offset)
    return u, gumbel(u)


def jitter_factors(num_tokens: int, width: int, eps: float, seed: int, offset: int) -> np.ndarray:
    """Multiplicative jitter f[s, c] = 1 + eps * (2u - 1), u ~ U(0, 1), in
    float32 arithmetic: each of 2u, 2u - 1, eps * (.), 1 + (.) rounded to the
    nearest float32 (reading R12).  Returned as float32."""
    u = stream_uniforms(num_tokens, width, PURPOSE_JITTER, seed, offset).astype(np.float32)
    two_u_m1 = (np.float32(2.0) * u) - np.float32(1.0)
    return np.float32(1.0) + np.float32(eps) * two_u_m1


def _feistel_bits(n: int) -> int:
    """Width of the Feistel domain: the smallest even b >= 2 with 2^b >= n."""
    b = 2
    while (1 << b) < n:
        b += 2
    return b


def rts_position(num_tokens: int, seed: int, offset: int) -> np.ndarray:
    """pi[s]: the queue position of token s under random token selection --
    a keyed pseudorandom permutation of 0..S-1 (reading R14): a 4-round
    Feistel network on b-bit words (halves of b/2 bits; round r maps the
    right half v to the left half XOR (word 0 of the RTS stream at index v,
    sub r, masked to b/2 bits)), restricted to [0, S) by cycle walking
    (applied again while the result is >= S)."""
    S = int(num_tokens)
    if S == 0:
        return np.zeros(0, dtype=np.int64)
    b = _feistel_bits(S)
    half = np.uint64(b // 2)
    mask = np.uint64((1 << (b // 2)) - 1)
    k0, k1 = _key(seed)
    off = int(offset) & 0xFFFFFFFFFFFFFFFF

    def perm(x):
        left, right = x >> half, x & mask
        for r in range(4):
            f = philox4x32_10(right, (PURPOSE_RTS << 24) | r, off & 0xFFFFFFFF, off >> 32,
                              k0, k1)[0] & mask
            left, right = right, left ^ f
        return (left << half) | right

    y = perm(np.arange(S, dtype=np.uint64))
    out_of_range = y >= np.uint64(S)
    while out_of_range.any():
        y[out_of_range] = perm(y[out_of_range])
        out_of_range = y >= np.uint64(S)
    return y.astype(np.int64)
