"""The near-tie validity check of the grouped-router GPU tests, on the CPU: it accepts the
oracle's own choices and rejects a choice outside the margin."""
import numpy as np
import pytest

from oracle import moe_oracle as om
from route_util import assert_valid_near_ties, decision_margins


def _case(seed=3, T=400, E=64, n_group=8):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((T, E)).astype(np.float32), (rng.standard_normal(E) * 0.2).astype(np.float32)


def test_validity_check_accepts_the_oracle_choices():
    logits, bias = _case()
    idx, _ = om.route_grouped(logits, 6, 8, 3, bias, 2.5)
    assert_valid_near_ties(idx, logits, 6, 8, 3, bias, 2e-6, np.arange(len(logits)))
    assert (decision_margins(logits, 6, 8, 3, bias) > 0).all()


def test_validity_check_rejects_a_wrong_expert_or_group():
    logits, bias = _case()
    idx, _ = om.route_grouped(logits, 6, 8, 3, bias, 2.5)
    t = 17
    bad = idx.copy()
    c = 1 / (1 + np.exp(-logits[t].astype(np.float64))) + bias
    gs = 8
    chosen_groups = set((idx[t] // gs).tolist())
    in_group = [e for e in range(64) if e // gs in chosen_groups and e not in idx[t]]
    bad[t, -1] = min(in_group, key=lambda e: c[e])          # the worst expert of an eligible group
    with pytest.raises(AssertionError):
        assert_valid_near_ties(bad, logits, 6, 8, 3, bias, 2e-6, [t])
    bad = idx.copy()
    other = [e for e in range(64) if e // gs not in chosen_groups]
    bad[t, -1] = max(other, key=lambda e: c[e])              # the best expert of a group not chosen
    with pytest.raises(AssertionError):
        assert_valid_near_ties(bad, logits, 6, 8, 3, bias, 2e-6, [t])
