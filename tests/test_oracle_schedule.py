"""Pins for the oracle's confidence calibration and prefix scheduler.

Source: "DSpark, la bozza che sa quando fermarsi" (paithon.it), section
"Verificare meglio, non di piu'": a_j = prod_{i<=j} c_i; the scheduler
admits candidate tokens of all requests in order of a_{r,j} while the
expected throughput Theta = tau * SPS(B) keeps growing, and stops at the first
candidate that does not raise it; temperature scaling keeps the ranking of
confidences and fixes only their magnitude.
"""
import itertools
import math

import numpy as np
import pytest
from scipy.special import expit

import oracle


def _sps(n_max, cap=512.0):
    return 1.0 / (1.0 + np.arange(n_max + 1) / cap)


def _theta(L, a, sps):
    tau = sum(1.0 + a[b, :L[b]].sum() for b in range(len(L)))
    btok = sum(l + 1 for l in L)
    return tau * sps[btok]


def test_calibration_identities():
    rng = np.random.default_rng(0)
    B, G = 6, 5
    cl = rng.normal(1, 1, (B, G))
    s = oracle.schedule(cl, np.ones(G), _sps(B * (G + 1)), 0, G)
    np.testing.assert_allclose(s["conf"], expit(cl), rtol=1e-14)
    np.testing.assert_allclose(s["cum_conf"], np.cumprod(expit(cl), axis=1), rtol=1e-13)
    # any positive per-position temperature keeps the ranking within a position
    T = np.linspace(1.0, 2.0, G)
    s2 = oracle.schedule(cl, T, _sps(B * (G + 1)), 0, G)
    for j in range(G):
        assert np.array_equal(np.argsort(cl[:, j], kind="stable"), np.argsort(s2["conf"][:, j], kind="stable"))
    np.testing.assert_allclose(s2["conf"], expit(cl / T), rtol=1e-14)


def test_greedy_early_stop_equals_brute_force_optimum():
    rng = np.random.default_rng(1)
    checked = 0
    for trial in range(300):
        B = int(rng.integers(1, 5))
        G = int(rng.integers(1, 4))
        L_min = int(rng.integers(0, G + 1))
        L_max = int(rng.integers(L_min, G + 1))
        cap = float(rng.choice([1.0, 4.0, 16.0, 512.0]))
        cl = rng.normal(1, 2, (B, G))
        sps = _sps(B * (L_max + 1), cap)
        s = oracle.schedule(cl, np.ones(G), sps, L_min, L_max)
        a = s["cum_conf"]
        best, arg = -1.0, None
        for L in itertools.product(range(L_min, L_max + 1), repeat=B):
            th = _theta(L, a, sps)
            if th > best + 1e-12:
                best, arg = th, L
        assert s["theta"] == pytest.approx(best, rel=1e-12)
        assert _theta(s["verify_len"], a, sps) == pytest.approx(s["theta"], rel=1e-12)
        if s["min_tie"] > 1e-9:
            assert tuple(s["verify_len"]) == arg
        checked += 1
    assert checked == 300


def test_admission_threshold_closed_form():
    # with SPS(n) = 1 / (1 + n / C): admitting a raises Theta iff a > tau / (C + n)
    rng = np.random.default_rng(2)
    B, G, C = 64, 5, 512.0
    cl = rng.normal(1, 1, (B, G))
    s = oracle.schedule(cl, np.linspace(1, 2, G), _sps(B * (G + 1), C), 1, G)
    a = s["cum_conf"]
    L = s["verify_len"]
    tau = sum(1.0 + a[b, :L[b]].sum() for b in range(B))
    n = int((L + 1).sum())
    admitted = [a[b, j] for b in range(B) for j in range(1, L[b])]
    rest = [a[b, j] for b in range(B) for j in range(L[b], G)]
    assert len(admitted) == s["n_admitted"]
    assert 1 <= L.min() and L.max() <= G and len(set(L.tolist())) > 1
    if rest:
        assert max(rest) <= tau / (C + n)
        assert min(admitted) > (tau - min(admitted)) / (C + n - 1)


def test_increasing_sps_admits_everything():
    rng = np.random.default_rng(3)
    B, G = 8, 4
    n = np.arange(B * (G + 1) + 1, dtype=float)
    sps = n / (1 + n / 512.0)   # read literally as steps/s, Theta only grows
    s = oracle.schedule(rng.normal(1, 1, (B, G)), np.ones(G), sps, 1, G)
    assert np.all(s["verify_len"] == G)


def test_step_shaped_sps_stops_at_first_drop():
    # Theta drops at the first admission but would rise later: the causal rule stops.
    B, G = 1, 3
    cl = np.full((B, G), 10.0)              # c ~ 1, a ~ 1
    sps = np.array([1.0, 1.0, 1.0, 0.5, 0.5])  # B_tok starts at 2 (L_min = 1)
    s = oracle.schedule(cl, np.ones(G), sps, 1, G)
    assert s["verify_len"].tolist() == [1] and s["n_admitted"] == 0
    # a table that dips only at 3 tokens: stops at 1 although 3 would be best
    sps2 = np.array([1.0, 1.0, 1.0, 0.6, 1.0])
    s2 = oracle.schedule(cl, np.ones(G), sps2, 1, G)
    assert s2["verify_len"].tolist() == [1]
    full = _theta([3], s2["cum_conf"], sps2)
    assert full > s2["theta"]


def test_candidate_order_ties_break_on_position_then_request():
    # equal confidences: a_{b,1} = 0.25 for every request; a table that allows
    # exactly one admission shows which candidate comes first (request 0)
    B, G = 3, 3
    cl = np.zeros((B, G))                    # c = 0.5
    sps = np.array([1.0] * 8 + [0.1] * 5)    # B_tok starts at 6; 7 keeps SPS, 8 drops it
    s = oracle.schedule(cl, np.ones(G), sps, 1, G)
    assert s["verify_len"].tolist() == [2, 1, 1] and s["n_admitted"] == 1
    # equal a across positions (c = 1 at position 1): the earlier position goes first
    cl2 = np.array([[0.0, 50.0, 0.0], [0.0, 0.0, 0.0], [0.0, 0.0, 0.0]])
    s2 = oracle.schedule(cl2, np.ones(G), sps, 0, G)
    # L_min = 0: B_tok starts at 3; SPS stays 1 up to 7 tokens -> four admissions:
    # a = 0.5 (b0 j0), 0.5 (b0 j1, tie broken by j), 0.5 (b1 j0), 0.5 (b2 j0)
    assert s2["verify_len"].tolist() == [2, 1, 1] and s2["n_admitted"] == 4
