"""Exhaustive-search statement of the group-limited top-k, for tiny inputs.

Independent of the oracle's sort-by-repeated-selection: it enumerates every
group subset and every expert subset and keeps the one with the largest exact
(rational) score sum, breaking ties by the lexicographically smallest sorted
index tuple.  For distinct values this is the same set as "the best by value";
for tied values the lexicographic rule keeps the lower indices, which is the
tie rule of the method (lower index wins).
"""
from fractions import Fraction
from itertools import combinations


def _best_subset(values, pool, size):
    best_key, best = None, None
    for sub in combinations(sorted(pool), size):
        total = sum(Fraction(float(values[i])) for i in sub)
        key = (total, tuple(-i for i in sub))  # larger sum, then smaller indices
        if best_key is None or key > best_key:
            best_key, best = key, sub
    return list(best)


def group_scores(s, n_groups):
    """Top-2 sum per group as the maximum pair sum over the group (FP32 add)."""
    import numpy as np
    gsize = len(s) // n_groups
    out = []
    for g in range(n_groups):
        members = [float(v) for v in s[g * gsize:(g + 1) * gsize]]
        if gsize == 1:
            out.append(np.float32(members[0]))
            continue
        out.append(max(np.float32(a) + np.float32(b)
                       for a, b in combinations(members, 2)))
    return out


def select(s, n_groups, topk_groups, top_k, scale):
    """-> (ids in slot order, weights, kept groups) for one token's scores s."""
    import numpy as np
    E = len(s)
    gsize = E // n_groups
    gs = group_scores(s, n_groups)
    kept = _best_subset(gs, range(n_groups), topk_groups)
    cand = [e for g in kept for e in range(g * gsize, (g + 1) * gsize)]
    chosen = _best_subset(list(s), cand, top_k)
    # slot order: score descending, expert ascending
    order = sorted(chosen, key=lambda e: (-Fraction(float(s[e])), e))
    S = np.float32(0.0)
    for e in order:
        S = np.float32(S + np.float32(s[e]))
    w = [np.float32(np.float32(np.float32(s[e]) / S) * np.float32(scale)) for e in order]
    return order, w, sorted(kept)
