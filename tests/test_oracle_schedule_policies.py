"""Pins of the oracle's other verify-length policies.

"DSpark, la bozza che sa quando fermarsi" (paithon.it), section "Che cosa resta
da verificare": the deployed scheduler works from confidences two rounds old
and drops the early stop; sections "Verificare meglio, non di piu'" and the
Chinese page's "置信度调度的验证" compare against a fixed confidence threshold.

Policy 1 (no early stop) must pick the global optimum of Theta = tau * SPS(B)
over every vector of verify lengths, for any SPS table: for a fixed number of
admitted positions the best set is the top-a one, which the shared candidate
order admits first.  That is checked by brute force.  The threshold policies
are pinned by their limits, by monotonicity in the threshold and by the
difference between a run (per-position c) and a count (non-increasing a).
"""
import itertools

import numpy as np
import pytest

import oracle


def _theta(L, a, sps):
    tau = sum(1.0 + a[b, :L[b]].sum() for b in range(len(L)))
    btok = sum(l + 1 for l in L)
    return tau * sps[btok]


def test_best_prefix_is_the_brute_force_optimum_for_any_table():
    rng = np.random.default_rng(11)
    for trial in range(300):
        B = int(rng.integers(1, 5))
        G = int(rng.integers(1, 4))
        L_min = int(rng.integers(0, G + 1))
        L_max = int(rng.integers(L_min, G + 1))
        cl = rng.normal(1, 2, (B, G))
        n = B * (L_max + 1) + 1
        kind = trial % 3
        if kind == 0:
            sps = 1.0 / (1.0 + np.arange(n) / float(rng.choice([2.0, 8.0, 512.0])))
        elif kind == 1:  # step-shaped: flat with drops
            sps = np.repeat(rng.uniform(0.2, 1.0, n // 2 + 1)[np.argsort(-rng.uniform(size=n // 2 + 1))], 2)[:n]
        else:            # arbitrary positive table
            sps = rng.uniform(0.1, 1.0, n)
        s = oracle.schedule_policy(cl, np.ones(G), sps, L_min, L_max, 1)
        a = s["cum_conf"]
        best, arg = -1.0, None
        for L in itertools.product(range(L_min, L_max + 1), repeat=B):
            th = _theta(L, a, sps)
            if th > best + 1e-12:
                best, arg = th, L
        assert s["theta"] == pytest.approx(best, rel=1e-12)
        assert _theta(s["verify_len"], a, sps) == pytest.approx(s["theta"], rel=1e-12)
        if s["min_margin"] > 1e-9 and s["min_tie"] > 1e-9:
            assert tuple(s["verify_len"]) == arg


def test_best_prefix_equals_early_stop_on_the_smooth_table():
    rng = np.random.default_rng(12)
    B, G = 40, 5
    sps = 1.0 / (1.0 + np.arange(B * (G + 1) + 1) / 512.0)
    for _ in range(20):
        cl = rng.normal(1, 1, (B, G))
        T = np.linspace(1.0, 2.0, G)
        e = oracle.schedule_policy(cl, T, sps, 1, G, 0)
        p = oracle.schedule_policy(cl, T, sps, 1, G, 1)
        assert np.array_equal(e["verify_len"], p["verify_len"])
        assert e["theta"] == pytest.approx(p["theta"], rel=1e-13)


def test_best_prefix_looks_past_a_dip_that_stops_the_early_rule():
    cl = np.full((1, 3), 10.0)
    sps = np.array([1.0, 1.0, 1.0, 0.6, 1.0])
    e = oracle.schedule_policy(cl, np.ones(3), sps, 1, 3, 0)
    p = oracle.schedule_policy(cl, np.ones(3), sps, 1, 3, 1)
    assert e["verify_len"].tolist() == [1]
    assert p["verify_len"].tolist() == [3]
    assert p["theta"] > e["theta"]


def test_threshold_on_survival_limits_and_monotonicity():
    rng = np.random.default_rng(13)
    B, G, L_min = 30, 6, 1
    cl = rng.normal(1, 1.5, (B, G))
    T = np.linspace(1.0, 2.0, G)
    sps = 1.0 / (1.0 + np.arange(B * (G + 1) + 1) / 512.0)
    lo = oracle.schedule_policy(cl, T, sps, L_min, G, 2, threshold=0.0)
    assert np.all(lo["verify_len"] == G)
    hi = oracle.schedule_policy(cl, T, sps, L_min, G, 2, threshold=1.0)
    assert np.all(hi["verify_len"] == L_min)
    prev = lo["verify_len"]
    for th in np.linspace(0.0, 1.0, 41):
        s = oracle.schedule_policy(cl, T, sps, L_min, G, 2, threshold=th)
        assert np.all(s["verify_len"] <= prev)
        prev = s["verify_len"]
        # a is non-increasing in j, so the run from L_min equals the count above th
        count = (s["cum_conf"][:, L_min:G] > th).sum(axis=1)
        assert np.array_equal(s["verify_len"] - L_min, count)
        assert _theta(s["verify_len"], s["cum_conf"], sps) == pytest.approx(s["theta"], rel=1e-12)
        assert s["n_admitted"] == int((s["verify_len"] - L_min).sum())


def test_threshold_on_confidence_is_a_leading_run():
    cl = np.array([[3.0, -3.0, 3.0, 3.0], [3.0, 3.0, 3.0, -3.0]])
    sps = np.ones(2 * 5 + 1)
    s = oracle.schedule_policy(cl, np.ones(4), sps, 0, 4, 3, threshold=0.5)
    # request 0 stops at its low second position although later ones are high
    assert s["verify_len"].tolist() == [1, 3]
    assert (s["conf"][0] > 0.5).sum() == 3
    near = oracle.schedule_policy(cl, np.ones(4), sps, 0, 4, 3, threshold=float(s["conf"][0, 0]))
    assert near["min_margin"] == 0.0   # a value on the threshold is reported as a tie
