"""Re-derive the Zipf bias strength ``ZIPF_KAPPA`` used by ``workloads.gen``.

The GLM-shaped workloads skew expert usage with a score-correction bias
b_e = -kappa * s * ln(rank(e)) (s = 1.1, ranks a seeded permutation), centred
to mean zero.  kappa is bisected once, on the 512-token prefill batch of seed
1004, until the busiest expert receives about 100 of the 512 tokens (the
workload's "0 to ~100" tokens per expert).  Routing uses the CPU oracle's
router, so no GPU code is involved.  Prints the kappa to freeze in gen.py.

    python -m workloads.calibrate_zipf
"""
from __future__ import annotations

import numpy as np

import oracle
from workloads import CONFIGS
from workloads.gen import gen_activations, gen_router


def busiest(kappa: float) -> tuple[int, np.ndarray]:
    w = CONFIGS["glm_prefill"]
    sh = w.shape
    x = gen_activations(w, 512, 0).float().numpy()
    rw, rb = gen_router(sh, w.seed, 0, "zipf", w.zipf_s, zipf_kappa=kappa)
    _, _, ids, _ = oracle.route(sh, rw.numpy(), rb.numpy(), x)
    c = np.bincount(ids.reshape(-1), minlength=sh.n_experts)
    return int(c.max()), c


def main(target: int = 100) -> float:
    lo, hi = 0.0, 0.08
    for _ in range(8):
        mid = 0.5 * (lo + hi)
        m, _ = busiest(mid)
        if m < target:
            lo = mid
        else:
            hi = mid
    kappa = round(0.5 * (lo + hi), 4)
    m, c = busiest(kappa)
    print(f"kappa={kappa} busiest={m} unused={(c == 0).sum()}")
    return kappa


if __name__ == "__main__":
    main()
