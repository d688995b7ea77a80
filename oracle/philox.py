"""Philox counter-based random numbers (oracle; test infrastructure only).

The pages need uniform random numbers for the acceptance coin and for
resampling ("Speculative Decoding", sections "The acceptance criterion" and "A
worked example") but fix no generator.  Philox is taken from Salmon, Moraes,
Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3" (SC'11): a keyed
bijection of a 4-word counter made of R rounds.  One round multiplies words 0
and 2 by fixed constants, keeps both halves of each product, mixes the high
halves with words 1 and 3 and the key, and permutes; the key is advanced by a
Weyl increment between rounds.

Written for any word width W in {32, 64} with Python integers, so that the
64-bit instance can be checked against NumPy's ``Philox`` (which is Philox4x64
with 10 rounds) and the 32-bit instance against the paper's known answers.
"""

_MULT = {32: (0xD2511F53, 0xCD9E8D57),
         64: (0xD2E7470EE14C6C93, 0xCA5A826395121157)}
_WEYL = {32: (0x9E3779B9, 0xBB67AE85),
         64: (0x9E3779B97F4A7C15, 0xBB67AE8584CAA73B)}


def philox4(counter, key, width=32, rounds=10):
    """Philox4xW-R of a 4-word counter under a 2-word key; returns 4 words."""
    mask = (1 << width) - 1
    m0, m1 = _MULT[width]
    w0, w1 = _WEYL[width]
    x0, x1, x2, x3 = (int(c) & mask for c in counter)
    k0, k1 = (int(k) & mask for k in key)
    for _ in range(rounds):
        p0 = m0 * x0
        p1 = m1 * x2
        hi0, lo0 = p0 >> width, p0 & mask
        hi1, lo1 = p1 >> width, p1 & mask
        x0, x1, x2, x3 = hi1 ^ x1 ^ k0, lo1, hi0 ^ x3 ^ k1, lo0
        k0 = (k0 + w0) & mask
        k1 = (k1 + w1) & mask
    return (x0, x1, x2, x3)


def philox4x32_10(counter, key):
    return philox4(counter, key, width=32, rounds=10)


def uniform_from_u32(x):
    """A 32-bit word to a uniform in [0, 1): its top 24 bits times 2**-24 (exact in fp32)."""
    return float(int(x) >> 8) * (2.0 ** -24)


def philox_uniform_pair(seed, offset, node, seq):
    """The two uniforms this library draws for (node, sequence) under (seed, offset).

    Key = (low, high) 32-bit halves of ``seed``; counter = (node, seq, low and
    high halves of ``offset``).  Word 0 gives the acceptance coin of the edge
    into ``node``; word 1 of node 0's block gives the sequence's resampling
    draw.  Returns (u0, u1).
    """
    seed = int(seed)
    offset = int(offset)
    key = (seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)
    ctr = (int(node), int(seq), offset & 0xFFFFFFFF, (offset >> 32) & 0xFFFFFFFF)
    w = philox4x32_10(ctr, key)
    return uniform_from_u32(w[0]), uniform_from_u32(w[1])


def acceptance_uniforms(seed, offset, B, T):
    """u_accept [B][T] (word 0 of block (c, b)) and u_sample [B] (word 1 of block (0, b))."""
    u_acc = [[0.0] * T for _ in range(B)]
    u_smp = [0.0] * B
    for b in range(B):
        for c in range(T):
            u0, u1 = philox_uniform_pair(seed, offset, c, b)
            u_acc[b][c] = u0
            if c == 0:
                u_smp[b] = u1
    return u_acc, u_smp
