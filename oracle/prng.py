"""Counter-based random numbers the method draws (test infrastructure only).

The pages say the rotation is a seeded random orthogonal matrix (Haar law,
intelliparadigm.com §2.1.1 step 1) and that QJL projects with a random
Gaussian matrix (same page §2.1.2); they do not fix a generator.  Reading
taken: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014, with the finaliser constants of Vigna's public
splitmix64.c), uniforms u = ((z >> 11) + 1) * 2^-53 in (0, 1], and standard
normals from the Box-Muller transform taken in pairs (cos first, then sin).

Pure Python integers: slow, but the path draws only d*d + m*d normals once.
"""
import math

_MASK = (1 << 64) - 1
_GAMMA = 0x9E3779B97F4A7C15


class SplitMix64:
    """SplitMix64: a Weyl sequence (step ``_GAMMA``) passed through a mixer."""

    def __init__(self, seed):
        self.state = seed & _MASK

    def next_u64(self):
        self.state = (self.state + _GAMMA) & _MASK
        z = self.state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK
        return z ^ (z >> 31)

    def next_uniform(self):
        """Uniform on (0, 1]: the top 53 bits plus one, times 2^-53."""
        return ((self.next_u64() >> 11) + 1) * (2.0 ** -53)


def gaussians(seed, count):
    """``count`` standard normals from one SplitMix64 stream (Box-Muller).

    Each pair (u1, u2) gives sqrt(-2 ln u1) * cos(2 pi u2) and then
    sqrt(-2 ln u1) * sin(2 pi u2); an odd count drops the last sine.
    """
    gen = SplitMix64(seed)
    out = []
    while len(out) < count:
        u1 = gen.next_uniform()
        u2 = gen.next_uniform()
        radius = math.sqrt(-2.0 * math.log(u1))
        angle = 2.0 * math.pi * u2
        out.append(radius * math.cos(angle))
        out.append(radius * math.sin(angle))
    return out[:count]
