"""Philox4x32-10 counter-based generator (oracle side).

Written from the generator's published definition (Salmon, Moraes, Dror,
Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC'11): ten rounds of
two 32x32->64 multiplies with constants 0xD2511F53 / 0xCD9E8D57, the key
bumped by the Weyl constants 0x9E3779B9 / 0xBB67AE85 between rounds.

The sampling verification draws its uniforms from it with
  key = (seed low word, seed high word),
  counter = (absolute position of the token being decided, draw index at that
             position, 0, 0),
  u = (first output word >> 8) * 2**-24, in [0, 1).
"""
M0, M1 = 0xD2511F53, 0xCD9E8D57
W0, W1 = 0x9E3779B9, 0xBB67AE85
MASK = 0xFFFFFFFF


def philox4x32_10(ctr, key):
    c0, c1, c2, c3 = (int(x) & MASK for x in ctr)
    k0, k1 = (int(x) & MASK for x in key)
    for r in range(10):
        if r:
            k0 = (k0 + W0) & MASK
            k1 = (k1 + W1) & MASK
        p0 = M0 * c0
        p1 = M1 * c2
        c0, c1, c2, c3 = ((p1 >> 32) ^ c1 ^ k0) & MASK, p1 & MASK, ((p0 >> 32) ^ c3 ^ k1) & MASK, p0 & MASK
    return [c0, c1, c2, c3]


def uniform(seed: int, position: int, draw: int) -> float:
    """The sampling draw for (position, draw index)."""
    x = philox4x32_10([position, draw, 0, 0], [seed & MASK, (seed >> 32) & MASK])
    return (x[0] >> 8) * (2.0 ** -24)
