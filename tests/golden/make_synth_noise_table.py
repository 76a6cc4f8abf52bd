"""Write the package's synth_noise_table.json: the MASK-row noise scale of
the synthetic model (``workloads.synth_rows``) per acceptance target.

Clean rows hold z with the generator's unit-variance values times
logit_std = 3 over V = 151936 entries; MASK rows hold z + sigma * e.  For
each target this script bisects sigma so that the mean over sample slots of
sum_v min(p_v, q_v) -- the probability that a draft drawn from q passes the
min(1, p/q) test -- equals the target, with both rows rounded to bfloat16 as
the generator stores them.  It calls only the oracle's softmax and the
workload generator.

    python tests/golden/make_synth_noise_table.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
from oracle.isd import softmax_t  # noqa: E402
from speculative_verify_accept_step_b300 import workloads as wl  # noqa: E402

V = 151936
LOGIT_STD = 3.0
SLOTS = 12
SEED = 4321
TARGETS = (0.5, 0.9, 0.99)


def rows(sigma):
    req = np.zeros(SLOTS, dtype=np.int64)
    pos = np.arange(SLOTS, dtype=np.int64) * 7 + 100
    sz, se = wl.synth_scale(LOGIT_STD), np.array([wl.synth_scale(sigma)], dtype=np.float32)
    p = wl.bf16_bits_to_f32(wl.synth_rows(req, pos, np.zeros(SLOTS, bool), V, sz, se, SEED, 0))
    q = wl.bf16_bits_to_f32(wl.synth_rows(req, pos, np.ones(SLOTS, bool), V, sz, se, SEED, 0))
    return p.astype(np.float64), q.astype(np.float64)


def mean_overlap(sigma):
    p, q = rows(sigma)
    return float(np.minimum(softmax_t(p, 1.0), softmax_t(q, 1.0)).sum(-1).mean())


def main():
    table = {}
    for t in TARGETS:
        lo, hi = 0.0, 8.0
        for _ in range(30):
            mid = 0.5 * (lo + hi)
            if mean_overlap(mid) > t:
                lo = mid
            else:
                hi = mid
        table[str(t)] = round(0.5 * (lo + hi), 6)
        print(t, table[str(t)], mean_overlap(table[str(t)]))
    out = dict(sigma=table, V=V, logit_std=LOGIT_STD, slots=SLOTS, seed=SEED,
               note="written by tests/golden/make_synth_noise_table.py")
    path = os.path.join(ROOT, "speculative_verify_accept_step_b300", "synth_noise_table.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
