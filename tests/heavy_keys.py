"""Choice of keys whose dK/dV gradients take the longest accumulations.

For each key the cost is the number of (query row, key) pairs the oracle
must visit to recompute the lse of every row that sees the key; within one
slice the rows that see key j are contiguous (the window [lo(r), hi(r)) of
every mask type is non-decreasing in the row r), so they are found by binary
search.  Keys seen by the most rows are the ones the dK/dV pass accumulates
over the most (q-tile, head) steps."""
import numpy as np

from oracle import planner


def key_rows(wl):
    """Number of query rows that see each key, and the per-slice row windows."""
    seen = np.zeros(wl.total_k, dtype=np.int64)
    for (qs, qe), (ks, ke), t in zip(wl.q_ranges, wl.k_ranges, wl.mask_types):
        if qe <= qs or ke <= ks:
            continue
        rows, lo, hi = planner.row_intervals(int(qs), int(qe), int(ks), int(ke), int(t))
        assert (np.diff(lo) >= 0).all() and (np.diff(hi) >= 0).all()
        j = np.arange(ks, ke)
        first = np.searchsorted(hi, j, side="right")  # first row with hi > j
        stop = np.searchsorted(lo, j, side="right")   # first row with lo > j
        seen[ks:ke] += np.maximum(stop - first, 0)
    return seen


def heaviest_keys(wl, n_top, n_random_prefix=0, prefix=None, seed=0):
    """The n_top keys seen by the most rows, taken from different slices'
    k ranges where possible, plus n_random_prefix random keys of [0, prefix)."""
    seen = key_rows(wl)
    picks = []
    order = np.argsort(-seen, kind="stable")
    used_ranges = set()
    for j in order:
        if len(picks) >= n_top or seen[j] == 0:
            break
        rng_id = next((i for i, (ks, ke) in enumerate(wl.k_ranges) if ks <= j < ke), -1)
        if rng_id in used_ranges:
            continue
        used_ranges.add(rng_id)
        picks.append(int(j))
    if n_random_prefix and prefix:
        rng = np.random.default_rng(seed)
        picks += [int(x) for x in rng.choice(prefix, n_random_prefix, replace=False)]
    return np.array(sorted(set(picks)), dtype=np.int64), seen
