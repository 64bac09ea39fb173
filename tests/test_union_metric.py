"""The host-side GQA reuse-rate measurement of bench.py against the oracle's PageWeaver union
(Sec. 2.2: U_G, membership masks, reuse rate rho_Q) on seeded random ordered masks."""
import numpy as np

import bench
from oracle import cosa_oracle as orc


def test_union_stats_match_oracle():
    rng = np.random.default_rng(12)
    B, H, nqb, pitch, G = 2, 8, 9, 6, 4
    mask = np.full((B, H, nqb, pitch), -1, np.int32)
    ml = np.zeros((B, H, nqb), np.int32)
    for b in range(B):
        for h in range(H):
            for i in range(nqb):
                k = int(rng.integers(1, min(pitch, i + 1) + 1))
                mask[b, h, i, :k] = rng.permutation(i + 1)[:k]
                ml[b, h, i] = k
    st = bench.union_stats(mask, ml, G)
    groups = [[list(mask[b, h, i, :ml[b, h, i]]) for h in range(g0, g0 + G)]
              for b in range(B) for g0 in range(0, H, G) for i in range(nqb)]
    assert abs(st["rho_Q"] - orc.reuse_rate(groups)) < 1e-12
    assert st["ordered_loads"] == sum(orc.ordered_shared_loads(gr) for gr in groups)
    assert st["union_blocks"] <= st["ordered_loads"] <= st["selections"]
