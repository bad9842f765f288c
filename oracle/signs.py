"""Random sign diagonal D of the rotation (oracle side; test infrastructure).

The Foundry spec ("TurboQuant KV Cache Compression — Spec", Algorithm Detail,
Step 1, and Lifecycle ``fa_tq_init(head_dim, config, seed)``) draws a
diagonal of random +1/-1 signs once from a seed but names no generator.
Reading: the generator is splitmix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014), a counter-based generator with
a published definition; output j (j = 0..d-1) gives sign j, and a set top bit
means D_jj = -1.  The CUDA library implements the same published generator
independently.
"""

import numpy as np

_MASK = (1 << 64) - 1
_GAMMA = 0x9E3779B97F4A7C15


def splitmix64(seed: int, count: int) -> list:
    """First ``count`` outputs of splitmix64 started from ``seed``.

    The state advances by the golden-ratio increment before each output; the
    output is the state passed through the variant-13 finaliser of
    MurmurHash3 (shifts 30, 27, 31 with the two published multipliers).
    """
    state = seed & _MASK
    outs = []
    for _ in range(count):
        state = (state + _GAMMA) & _MASK
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK
        outs.append(z ^ (z >> 31))
    return outs


def sign_diagonal(seed: int, d: int = 128) -> np.ndarray:
    """Diagonal of D as float64 +1/-1 values (top bit of output j set => -1)."""
    return np.array([-1.0 if (o >> 63) else 1.0 for o in splitmix64(seed, d)],
                    dtype=np.float64)
