"""Write the package's noise_table.json: the MASK-logit noise scale per
acceptance target (input-generation data that the seeded workloads read).

The synthetic q-logits of a draft are the verifying row's clean logits z plus
sigma * N(0, 1).  For z ~ N(0, 3^2) over V = 151936 entries (both rows rounded
to bfloat16, as the workloads store them) this script bisects sigma so that the
mean over sample rows of sum_v min(p_v, q_v) -- the probability that a draft
drawn from q passes the min(1, p/q) test -- equals each target.  It calls only
the oracle's softmax.

    python tests/golden/make_noise_table.py
"""
import json
import os
import sys

import numpy as np
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))
from oracle.isd import softmax_t  # noqa: E402

V = 151936
LOGIT_STD = 3.0
ROWS = 16
SEED = 1234
TARGETS = (0.5, 0.9, 0.99)


def mean_overlap(z, eps, sigma):
    y = torch.from_numpy(z + sigma * eps).bfloat16().double().numpy()
    return float(np.minimum(softmax_t(z, 1.0), softmax_t(y, 1.0)).sum(-1).mean())


def main():
    g = torch.Generator().manual_seed(SEED)
    z = (torch.randn(ROWS, V, generator=g) * LOGIT_STD).bfloat16().double().numpy()
    eps = torch.randn(ROWS, V, generator=g).double().numpy()
    table = {}
    for t in TARGETS:
        lo, hi = 0.0, 8.0
        for _ in range(40):
            mid = 0.5 * (lo + hi)
            if mean_overlap(z, eps, mid) > t:
                lo = mid
            else:
                hi = mid
        table[str(t)] = round(0.5 * (lo + hi), 6)
        print(t, table[str(t)], mean_overlap(z, eps, table[str(t)]))
    out = dict(sigma=table, V=V, logit_std=LOGIT_STD, rows=ROWS, seed=SEED,
               note="written by tests/golden/make_noise_table.py")
    root = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    path = os.path.join(root, "speculative_verify_accept_step_b300", "noise_table.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
