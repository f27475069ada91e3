"""Decision margins and near-tie validity of the group-limited sigmoid router, for GPU tests.

The router decides in fp32 on both sides, but the GPU's and NumPy's sigmoids may round
differently in the last bit.  Indices are therefore compared bit for bit on tokens whose
group cut and expert cut clear a margin of a few fp32 ulps, and every other token's choice
is checked to be one an exact-arithmetic router could make within that margin.
"""
import numpy as np


def selection_scores(logits, bias):
    """c = sigmoid(l) + bias in fp32, as both sides compute it (up to the last bit)."""
    one = np.float32(1.0)
    return (one / (one + np.exp(-logits.astype(np.float32)))) + bias.astype(np.float32)[None, :]


def group_scores(c, n_group):
    """Sum of the two largest c of each group of E / n_group consecutive experts, [T, n_group]."""
    T, E = c.shape
    top2 = -np.sort(-c.reshape(T, n_group, E // n_group), axis=2)[:, :, :2]
    return (top2[:, :, 0].astype(np.float64) + top2[:, :, 1])


def eligible_groups(c, n_group, topk_group):
    """[T, n_group] mask of the topk_group best groups (ties to the lower group)."""
    T = c.shape[0]
    gsc = group_scores(c, n_group)
    order = np.lexsort((np.broadcast_to(np.arange(n_group), (T, n_group)), -gsc), axis=-1)
    el = np.zeros((T, n_group), bool)
    np.put_along_axis(el, order[:, :topk_group], True, axis=1)
    return el


def _cuts(c, k, n_group, topk_group):
    """Per token: the topk_group-th best group score and the k-th best c among the experts of
    the eligible groups, and the gaps to the next candidates at both cuts."""
    T, E = c.shape
    gs = E // n_group
    gsc = np.sort(group_scores(c, n_group), axis=1)[:, ::-1]
    g_cut = gsc[:, topk_group - 1]
    g_gap = g_cut - gsc[:, topk_group] if topk_group < n_group else np.full(T, np.inf)
    eligible_c = np.where(np.repeat(eligible_groups(c, n_group, topk_group), gs, axis=1), c, -np.inf)
    cs = np.sort(eligible_c.astype(np.float64), axis=1)[:, ::-1]
    e_cut = cs[:, k - 1]
    e_gap = e_cut - cs[:, k] if k < topk_group * gs else np.full(T, np.inf)
    return g_cut, g_gap, e_cut, e_gap


def decision_margins(logits, k, n_group, topk_group, bias):
    """Per token: the smaller of the gaps at the group cut and at the expert cut."""
    _, g_gap, _, e_gap = _cuts(selection_scores(logits, bias), k, n_group, topk_group)
    return np.minimum(g_gap, e_gap)


def assert_valid_near_ties(idx, logits, k, n_group, topk_group, bias, margin, tokens):
    """For each given token: k distinct experts from at most topk_group groups, every chosen
    group's score within `margin` of the group cut, and every chosen expert's c within
    `margin` of the k-th best c among the eligible groups' experts."""
    c = selection_scores(logits[tokens], bias)
    g_cut, _, e_cut, _ = _cuts(c, k, n_group, topk_group)
    gsc = group_scores(c, n_group)
    gs = logits.shape[1] // n_group
    for i, t in enumerate(tokens):
        chosen = idx[t]
        assert len(set(chosen.tolist())) == k, (t, chosen)
        groups = set((chosen // gs).tolist())
        assert len(groups) <= topk_group, (t, chosen)
        for g in groups:
            assert gsc[i, g] >= g_cut[i] - margin, (t, g, gsc[i, g], g_cut[i])
        for e in chosen:
            assert c[i, e] >= e_cut[i] - margin, (t, e, c[i, e], e_cut[i])
