"""Selection inputs with exact ties, and the expected ids worked out by hand
from the tie rules ("GLM-5.2 on a 32 GB Mac - native MLX port of the Colibri
hierarchy", "G2 implementation status": lower expert id on an exact tie; tied
group scores go to the lower group index).  Used by the GPU tie tests and
checked against the oracle on the CPU."""
from __future__ import annotations

import numpy as np

def tie_bias(E: int, n_group: int, kind: str) -> np.ndarray:
    """Biases b with keys 0.5 + b exact in fp32 (binary fractions).

    kth    four kept groups hold three experts each at key 0.75 (twelve exact
           ties for the last seven places behind one expert at key 1.0); the
           other groups hold one such expert, so their score is lower
    groups two groups score 2.0, five groups tie at 1.5 for the remaining
           two kept places (the lower group indices must win), one scores 0.5
    equal  every key 0.5: the k lowest ids, all groups tied
    """
    gs = E // n_group
    b = np.full(E, -0.25, np.float32)  # key 0.25
    if kind == "equal":
        return np.zeros(E, np.float32)
    if kind == "kth":
        for g in range(n_group):
            pos = (2, 5, 9) if g in (1, 3, 4, 6) else (7,)
            for p in pos:
                b[g * gs + p % gs] = 0.25   # key 0.75
        b[4 * gs + 20 % gs] = 0.5           # key 1.0 in group 4
        return b
    if kind == "groups":
        for g in (2, 5):
            b[g * gs + 1 % gs] = 0.5
            b[g * gs + 11 % gs] = 0.5       # score 2.0
        for g in (0, 1, 3, 4, 6):
            b[g * gs + 3 % gs] = 0.25
            b[g * gs + 17 % gs] = 0.25      # score 1.5: five groups tied
        return b
    raise ValueError(kind)


KINDS = ("kth", "groups", "equal")


def expected_ids_t1(kind, E, n_group, k):
    gs = E // n_group
    if kind == "equal":
        return list(range(k))
    if kind == "kth":
        top = [4 * gs + 20 % gs]
        tied = sorted(g * gs + p % gs for g in (1, 3, 4, 6) for p in (2, 5, 9))
        return top + tied[:k - 1]
    if kind == "groups":
        hi = [g * gs + p % gs for g in (2, 5) for p in (1, 11)]
        mid = [g * gs + p % gs for g in (0, 1) for p in (3, 17)]
        return sorted(hi) + sorted(mid)
    raise ValueError(kind)
