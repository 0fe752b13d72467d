"""Fragile-layer selection after a profiling window (GIFT reading notes, simplification 3 and
Figure 3): scores from window-summed boundary-hit counts, ranking, and the cut at the knee.

The oracle's rule is pinned on hand-built score curves whose answer is fixed by inspection.
The library's host function (gift_select_fragile, no GPU involved) is then compared with the
oracle on seeded random windows: the full ranking, the scores bit for bit (both sides divide
the same integers in double) and the selected count."""
import math

import numpy as np
import pytest

import oracle as O
from fac_whitening_gb300 import gift as G


def _lib_or_skip():
    try:
        return G.lib()
    except RuntimeError as e:  # not built in this checkout
        pytest.skip(str(e))


def counts_for(scores, n):
    """Window counts whose score is the nearest multiple of 1/n: lower hits carry it, with
    one upper hit per layer (the amax element lands on the largest code)."""
    return [(1, int(round(s * n)) - 1, n) for s in scores]


# ---- the oracle's rule, pinned --------------------------------------------------------

def test_knee_figure3_shape():
    # 48 MLP layers: a fragile group of 13 (scores 0.12 .. 0.08), then a clear drop to the
    # rest (0.02 .. 0.005), in a shuffled layer order: the knee selects exactly the group
    rng = np.random.default_rng(3)
    high, low = np.linspace(0.12, 0.08, 13), np.linspace(0.02, 0.005, 35)
    perm = rng.permutation(48)
    scores = np.empty(48)
    scores[perm[:13]], scores[perm[13:]] = high, low
    sel = O.select_fragile_knee(list(scores))
    assert sorted(sel) == sorted(perm[:13].tolist())
    assert O.knee_count(sorted(scores, reverse=True)) == 13


def test_knee_rule_cases():
    assert O.knee_count([0.5]) == 1                                # one layer
    assert O.knee_count([0.1] * 5) == 1                            # no drop anywhere: the smallest k
    assert O.knee_count([0.5, 0.375, 0.25, 0.125]) == 1            # equal (dyadic) drops: the smaller k
    assert O.knee_count([0.9, 0.1, 0.09, 0.01]) == 1
    assert O.knee_count([0.9, 0.1, 0.09, 0.01], k_min=2) == 3      # searched from k_min
    assert O.knee_count([0.9, 0.8, 0.1, 0.0], k_max=1) == 1        # and up to k_max
    assert O.knee_count([0.3, 0.2, 0.1], k_min=3) == 3             # k_min = L: all layers
    with pytest.raises(ValueError):
        O.knee_count([0.3, 0.2], k_min=2, k_max=1)


def test_window_score_is_the_mean_rate():
    # summed counts over the summed n equal the mean of the per-step rates (n fixed per step)
    rng = np.random.default_rng(4)
    n = 1536 * 6144
    steps = [(int(rng.integers(0, 50)), int(rng.integers(0, 5000)), n) for _ in range(100)]
    window = tuple(sum(c[i] for c in steps) for i in range(3))
    mean_rate = sum(O.fragility_score(c) for c in steps) / len(steps)
    assert math.isclose(O.window_scores([window])[0], mean_rate, rel_tol=1e-12)


def test_fixed_k_matches_plain_ranking():
    scores = [0.1, 0.3, 0.3, 0.05, 0.2]
    assert O.select_fragile(scores, 3) == [1, 2, 4]
    assert O.select_fragile_knee(scores, k_min=3, k_max=3) == [1, 2, 4]


# ---- libgift's host function against the oracle ----------------------------------------

def _random_window(rng):
    L = int(rng.integers(1, 61))
    n_step = int(rng.choice([1536 * 1536, 1536 * 6144, 777]))
    steps = int(rng.integers(1, 101))
    n = n_step * steps
    rows = []
    for _ in range(L):
        kind = rng.integers(0, 4)
        if kind == 0:
            rows.append((0, 0, n))                                    # no hits
        elif kind == 1 and rows:
            rows.append(rows[int(rng.integers(0, len(rows)))])        # a tie with an earlier layer
        else:
            rows.append((int(rng.integers(0, steps * 4 + 1)), int(rng.integers(0, n // 10 + 1)), n))
    return rows


def test_library_matches_oracle_on_random_windows():
    _lib_or_skip()
    rng = np.random.default_rng(5)
    for _ in range(300):
        rows = _random_window(rng)
        L = len(rows)
        want_scores = O.window_scores(rows)
        want_order = sorted(range(L), key=lambda i: (-want_scores[i], i))
        k = int(rng.integers(0, L + 1))
        k_min = int(rng.integers(1, L + 1))
        k_max = int(rng.integers(k_min, L + 1))
        order, scores, k_out = G.gift_select_fragile(rows, k=k, k_min=k_min, k_max=k_max)
        assert scores == want_scores
        assert order == want_order
        want_k = k if k > 0 else O.knee_count([want_scores[i] for i in want_order], k_min, k_max)
        assert k_out == want_k
        if k == 0:
            assert order[:k_out] == O.select_fragile_knee(want_scores, k_min, k_max)


def test_library_figure3_shape_and_dyadic_ties():
    _lib_or_skip()
    n = 1536 * 6144 * 100
    scores = list(np.linspace(0.12, 0.08, 13)) + list(np.linspace(0.02, 0.005, 35))
    order, _, k = G.gift_select_fragile(counts_for(scores, n))
    assert k == 13 and sorted(order[:13]) == list(range(13))
    # equal drops between dyadic scores: the smaller k
    order, scores, k = G.gift_select_fragile([(0, 2, 8), (0, 4, 8), (0, 1, 8), (0, 3, 8)])
    assert scores == [0.25, 0.5, 0.125, 0.375] and order == [1, 3, 0, 2] and k == 1


def test_library_rejects_bad_arguments():
    _lib_or_skip()
    rows = [(1, 2, 100), (0, 5, 100), (3, 0, 100)]
    for kwargs in ({"k": 4}, {"k": -1}, {"k": 0, "k_min": 0}, {"k": 0, "k_min": 3, "k_max": 2},
                   {"k": 0, "k_max": 4}):
        with pytest.raises(G.GiftError):
            G.gift_select_fragile(rows, **kwargs)
    with pytest.raises(G.GiftError):
        G.gift_select_fragile([(101, 0, 100)])     # more hits than elements
    with pytest.raises(G.GiftError):
        G.gift_select_fragile([])                   # no layers


def test_window_of_heavy_tailed_layers_end_to_end():
    # a 5-step profiling window over 12 heavy-tailed layers (the profiler workload's kind of
    # tensor, small shapes; half the layers with a much wider column spread, the "fragile"
    # ones): counts summed with the oracle's boundary-hit rule, then the library's selection
    # must equal the oracle's, in both formats
    _lib_or_skip()
    from fac_whitening_gb300 import synth
    for fmt in ("e4m3", "e5m2"):
        window = [[0, 0, 0] for _ in range(12)]
        for step in range(5):
            for layer in range(12):
                spread = 4.0 if layer % 2 else 1.0
                W = synth.student_t_colscaled(48, 64, seed=1000 * step + layer, col_sigma=spread).numpy()
                up, lo, n = O.boundary_hits(W, fmt)
                window[layer][0] += up
                window[layer][1] += lo
                window[layer][2] += n
        order, scores, k = G.gift_select_fragile(window)
        want = O.window_scores(window)
        assert scores == want
        assert order[:k] == O.select_fragile_knee(want)
        assert k >= 1 and all(s > 0 for s in scores)
        if fmt == "e4m3":   # E4M3's narrow range: the knee picks exactly the wide-spread layers
            assert sorted(order[:k]) == [1, 3, 5, 7, 9, 11]
