"""Philox4x32-10, written from its published definition.

Reference: J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel
random numbers: as easy as 1, 2, 3", SC'11 (the Philox-4x32 bijection with
R = 10 rounds).  One round maps the counter (c0, c1, c2, c3) under the round
key (k0, k1) to

    (hi(M1*c2) ^ c1 ^ k0,  lo(M1*c2),  hi(M0*c0) ^ c3 ^ k1,  lo(M0*c0))

with M0 = 0xD2511F53, M1 = 0xCD9E8D57; between rounds the key is bumped by
the Weyl constants (0x9E3779B9, 0xBB67AE85) modulo 2^32.

Also holds the three *uses* of the generator by the decoder (each a stated
reading; the pages do not fix how random numbers are drawn):

  * canvas initialisation, x_1 ~ Unif(V^C) (report §2.1): position i of
    canvas k takes word 0 of Philox(key=seed, ctr=(i, 0, k, TAG_INIT)) and
    maps it to floor(word * V / 2^32);
  * the Gumbel noise of the re-noise step: vocab entry v of position i at
    step n of canvas k uses word (v mod 4) of
    Philox(key=seed, ctr=(v div 4, i, (k << 16) | n, TAG_GUMBEL)), turned into
    the open-interval uniform u = (2*(word >> 9) + 1) * 2^-24;
  * synthetic weights (see oracle.weights): element e of tensor t uses
    Philox(key=weight_seed, ctr=(e mod 2^32, e div 2^32, t, TAG_WEIGHT)).

parity pinned by: tests/test_oracle_philox.py (Random123 known-answer
vectors, uniformity chi-square of the init ids).
"""
import numpy as np

_M0 = np.uint64(0xD2511F53)
_M1 = np.uint64(0xCD9E8D57)
_W0 = np.uint64(0x9E3779B9)
_W1 = np.uint64(0xBB67AE85)
_LO = np.uint64(0xFFFFFFFF)
_S32 = np.uint64(32)

TAG_WEIGHT = 1
TAG_INIT = 2
TAG_GUMBEL = 3


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Apply the 10-round Philox-4x32 bijection elementwise.

    Counters and keys are (broadcastable) unsigned 32-bit integers; returns
    the four output words as uint32 arrays.
    """
    c0, c1, c2, c3 = (np.asarray(c, dtype=np.uint64) & _LO for c in (c0, c1, c2, c3))
    k0 = np.asarray(k0, dtype=np.uint64) & _LO
    k1 = np.asarray(k1, dtype=np.uint64) & _LO
    for _ in range(10):
        p0 = _M0 * c0          # < 2^64: exact in uint64
        p1 = _M1 * c2
        c0, c1, c2, c3 = ((p1 >> _S32) ^ c1 ^ k0,
                          p1 & _LO,
                          (p0 >> _S32) ^ c3 ^ k1,
                          p0 & _LO)
        k0 = (k0 + _W0) & _LO
        k1 = (k1 + _W1) & _LO
    return tuple(w.astype(np.uint32) for w in (c0, c1, c2, c3))


def split_seed(seed):
    """64-bit seed -> Philox key (low word, high word)."""
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    return seed & 0xFFFFFFFF, seed >> 32


def canvas_init_ids(seed, k, canvas_len, vocab):
    """x_1 of canvas k: C ids, each uniform over the vocabulary (report §2.1)."""
    k0, k1 = split_seed(seed)
    i = np.arange(canvas_len, dtype=np.uint64)
    w0, _, _, _ = philox4x32_10(i, 0, k, TAG_INIT, k0, k1)
    return ((w0.astype(np.uint64) * np.uint64(vocab)) >> _S32).astype(np.int32)


def gumbel_uniforms(seed, k, n, positions, vocab):
    """Open-interval fp32 uniforms u[len(positions), vocab] for step n of canvas k."""
    k0, k1 = split_seed(seed)
    pos = np.asarray(positions, dtype=np.uint64)[:, None]
    quad = np.arange(vocab // 4, dtype=np.uint64)[None, :]
    ctr2 = (int(k) << 16) | int(n)
    words = philox4x32_10(quad, pos, ctr2, TAG_GUMBEL, k0, k1)
    w = np.stack(words, axis=-1).reshape(len(positions), vocab)   # v = 4*quad + word
    odd = ((w >> np.uint32(9)).astype(np.int64) * 2 + 1).astype(np.float32)  # < 2^24: exact
    return odd * np.float32(2.0 ** -24)
