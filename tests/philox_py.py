"""Independent pure-Python Philox4x32-10 used by the tests to pin the oracle's
and the library's random streams. Written from Salmon et al., "Parallel Random
Numbers: As Easy as 1, 2, 3" (SC'11); checked against the published
known-answer vectors in tests/golden/philox4x32_10_kat.txt."""
import numpy as np

MULT = (0xD2511F53, 0xCD9E8D57)
WEYL = (0x9E3779B9, 0xBB67AE85)
MASK = 0xFFFFFFFF


def philox(ctr, key, rounds=10):
    x0, x1, x2, x3 = (int(c) & MASK for c in ctr)
    k0, k1 = (int(k) & MASK for k in key)
    for r in range(rounds):
        if r:
            k0, k1 = (k0 + WEYL[0]) & MASK, (k1 + WEYL[1]) & MASK
        a = MULT[0] * x0
        c = MULT[1] * x2
        x0, x1, x2, x3 = (c >> 32) ^ x1 ^ k0, c & MASK, (a >> 32) ^ x3 ^ k1, a & MASK
    return x0, x1, x2, x3


def philox_vec(c0, c1, c2, c3, k0, k1, rounds=10):
    """Vectorised over numpy uint32 counter arrays (uint64 arithmetic)."""
    x0, x1, x2, x3 = (np.asarray(c, dtype=np.uint64) for c in (c0, c1, c2, c3))
    k0 = np.uint64(k0)
    k1 = np.uint64(k1)
    m = np.uint64(MASK)
    for r in range(rounds):
        if r:
            k0 = (k0 + np.uint64(WEYL[0])) & m
            k1 = (k1 + np.uint64(WEYL[1])) & m
        a = np.uint64(MULT[0]) * x0
        c = np.uint64(MULT[1]) * x2
        x0, x1, x2, x3 = (c >> np.uint64(32)) ^ x1 ^ k0, c & m, (a >> np.uint64(32)) ^ x3 ^ k1, a & m
    return tuple(v.astype(np.uint32) for v in (x0, x1, x2, x3))


def accept_uniform(seed, b, j):
    x = philox((b, j, 0, 1), (seed & MASK, seed >> 32))[0]
    return np.float32(x >> 8) * np.float32(2.0 ** -24)


def race_words_vec(seed, b, j, v, tag):
    """Race word of vocabulary index v: word v % 4 of counter (b, j, v // 4, tag)."""
    v = np.asarray(v, dtype=np.uint64)
    words = philox_vec(np.full_like(v, b), np.full_like(v, j), v >> np.uint64(2), np.full_like(v, tag), seed & MASK,
                       seed >> 32)
    return np.choose((v & np.uint64(3)).astype(np.int64), words)


def race_exponential_vec(seed, b, j, v, tag):
    """E = -log1p(-u), u = float32(x) * 2^-32 of the race word x, in float32 (numpy)."""
    x = race_words_vec(seed, b, j, v, tag)
    u = x.astype(np.float32) * np.float32(2.0 ** -32)
    return -np.log1p(-u)
