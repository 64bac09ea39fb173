"""Plant plausible mistakes in copies of the oracle and check that the pins catch each one.

Every mutation is a one-token edit of the oracle's source (a dropped term, a wrong
sign, index or comparison); the test runs the pins of ``oracle_checks`` on the
mutated module and expects at least one to fail.
"""
import inspect
import sys
import types

import pytest

from oracle import cosa_oracle
from tests import oracle_checks as oc

MUTATIONS = {
    # OSK (Algorithm A)
    "skip_vs_previous_max": ("diff = np.where(has, m_loc - np.where(has, m, 0.0), -np.inf)",
                             "diff = np.where(has, m_loc - np.where(has, m_prev, 0.0), -np.inf)"),
    "vote_min_over_rows": ("worst = diff.max()", "worst = diff.min()"),
    "skip_le_instead_of_lt": ("skip = worst < tau", "skip = worst <= tau"),
    "no_scale_in_osk": ("S = (Qi @ K[c0:c1].T) * prm.sm_scale", "S = (Qi @ K[c0:c1].T)"),
    "no_causal_in_osk": ("vis = (keys_pos[None, :] <= rows_pos[:, None]) & exists[c0:c1][None, :]",
                         "vis = (keys_pos[None, :] >= 0) & exists[c0:c1][None, :]"),
    "no_rescale": ("l = alpha * l + Pt.sum(axis=1)", "l = l + Pt.sum(axis=1)"),
    "duplicates_kept": ("if j < 0 or j > i or j >= nblk or j in seen:", "if j < 0 or j > i or j >= nblk:"),
    "future_blocks_kept": ("if j < 0 or j > i or j >= nblk or j in seen:", "if j < 0 or j >= nblk or j in seen:"),
    "threshold_uses_total_not_delta": ("tau = math.log(prm.skip_delta / L) if use_skip else 0.0",
                                       "tau = math.log(1.0 / L) if use_skip else 0.0"),
    "missing_page_kept": ("vis = (keys_pos[None, :] <= rows_pos[:, None]) & exists[c0:c1][None, :]",
                          "vis = (keys_pos[None, :] <= rows_pos[:, None])"),
    # token set
    "token_set_strict_causal": ("return [t for t in range(0, L) if (t // P) in S and t <= c]",
                                "return [t for t in range(0, L) if (t // P) in S and t < c]"),
    # KAP (Eqs. 8-14)
    "maxpool_is_mean": ("Pm[:, j] = S_hat[:, starts[j]:ends[j]].max(axis=1)",
                        "Pm[:, j] = S_hat[:, starts[j]:ends[j]].mean(axis=1)"),
    "no_maxnorm": ("return np.where(pmax > 0, Pm / np.where(pmax > 0, pmax, 1.0), 0.0)",
                   "return Pm"),
    "kap_not_causal": ("visible = (keys_pos[None, :] <= rows_pos[:, None]) & ks_exists[None, :]",
                       "visible = ks_exists[None, :] & (keys_pos[None, :] >= 0)"),
    "hrm_threshold_loose": ("hrm = (pbar == 1.0).any(axis=0)", "hrm = (pbar >= 0.5).any(axis=0)"),
    "sort_ascending": ("H = H[np.lexsort((H, -scores[H]))]", "H = H[np.lexsort((H, scores[H]))]"),
    "rest_sort_ascending": ("R = R[np.lexsort((R, -scores[R]))]", "R = R[np.lexsort((R, scores[R]))]"),
    "tie_break_descending": ("R = R[np.lexsort((R, -scores[R]))]", "R = R[np.lexsort((-R, -scores[R]))]"),
    "no_hrm_first": ("return np.concatenate([H, R]).astype(np.int64)",
                     "return np.concatenate([H, R])[np.lexsort((np.concatenate([H, R]), -scores[np.concatenate([H, R])]))].astype(np.int64)"),
    "budget_floor": ("return max(1, min(J, -(-budget_ppm * J // 1_000_000)))",
                     "return max(1, min(J, budget_ppm * J // 1_000_000))"),
    "no_scale_in_kap": ("logits = (Qs_rows @ Ks.T) * sm_scale", "logits = (Qs_rows @ Ks.T)"),
    # ablation modes
    "ascending_left_unsorted": ("mask[bi, h, i, :row.K] = np.sort(sel) if ascending else sel",
                                "mask[bi, h, i, :row.K] = sel"),
    "ascending_sorts_before_truncation": ("sel = row.order[:row.K]", "sel = np.sort(row.order)[:row.K]"),
    "binary_flags_by_visit": ("flags[j] = r.flags[x]", "flags[x] = r.flags[x]"),
    "binary_walk_includes_diagonal_only": ("walk = min(n, i + 1)", "walk = min(n, i)"),
    "binary_mask_keeps_future": ("if 0 <= j <= i:", "if 0 <= j:"),
    # top-p stage-1 length
    "top_p_strict": ("return int(np.argmax(csum >= thr)) + 1", "return int(np.argmax(csum > thr)) + 1"),
    "top_p_score_order": ("csum = np.cumsum(scores[order])", "csum = np.cumsum(np.sort(scores)[::-1])"),
    "top_p_off_by_one": ("return int(np.argmax(csum >= thr)) + 1", "return max(1, int(np.argmax(csum >= thr)))"),
    # PageWeaver union and reuse rate
    "reuse_rate_counts_repeats": ("num = sum(len(set(int(x) for x in S)) for G in groups for S in G)",
                                  "num = sum(len(S) for G in groups for S in G)"),
    "shared_load_serves_one_head": ("                pos[h] += 1\n", "                pos[h] += 1\n                break\n"),
    "union_tie_to_highest_id": ("blk = min(cand, key=lambda b: (-cand[b], b))", "blk = min(cand, key=lambda b: (-cand[b], -b))"),
    "union_fewest_heads_first": ("blk = min(cand, key=lambda b: (-cand[b], b))", "blk = min(cand, key=lambda b: (cand[b], b))"),
    "kept_visits_keeps_future": ("if not (0 <= j <= i and j < nblk) or j in seen:", "if not (0 <= j and j < nblk) or j in seen:"),
    "kept_visits_keeps_repeats": ("if not (0 <= j <= i and j < nblk) or j in seen:", "if not (0 <= j <= i and j < nblk):"),
}


def _mutant(name):
    old, new = MUTATIONS[name]
    src = inspect.getsource(cosa_oracle)
    assert src.count(old) == 1, f"mutation target not unique or missing: {name}"
    mod = types.ModuleType(f"oracle_mutant_{name}")
    sys.modules[mod.__name__] = mod          # dataclasses resolve annotations through sys.modules
    try:
        exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), mod.__dict__)
    finally:
        sys.modules.pop(mod.__name__, None)
    return mod


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name):
    mod = _mutant(name)
    caught = []
    for check in oc.ALL_CHECKS:
        try:
            check(mod)
        except Exception:  # an assertion or any error in the mutant counts as caught
            caught.append(check.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
