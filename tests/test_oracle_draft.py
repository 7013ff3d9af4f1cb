"""Pins for the oracle's draft sampler (semi-autoregressive Markov head).

Sources: "DSpark, la bozza che sa quando fermarsi" (paithon.it), section
"Un po' di autoregressione basta": the draft distribution at position k is
softmax(U_k + B_k) with the Markov bias B = W1 W2 driven by the previous
token, and the block is sampled left to right.

The draw is per-token Gumbel-max: x = argmax_v (s_v + g(u_v)) with u_v the
token's own Philox word (counter (v >> 2, j, request, stream 0), word v & 3).
Its pins: on constant rows the key order is the order of the uniforms, so the
token is the argmax of the token uniforms (lowest id on ties), and over 10^6
draws the token frequencies follow softmax(s) (chi-square), on a tiny and on
a 40-token vocabulary.
"""
import math

import numpy as np
import pytest

import oracle


def _chi2_ok(counts, probs, n, sigmas=6.0):
    exp = probs * n
    mask = exp > 0
    chi2 = (((counts - exp) ** 2)[mask] / exp[mask]).sum()
    dof = mask.sum() - 1
    return chi2 < dof + sigmas * math.sqrt(2 * dof), chi2


def _softmax(x):
    e = np.exp(x - x.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def test_constant_row_closed_form():
    V, r = 1000, 4
    U = np.full((1, 1, V), 2.5)
    E = np.zeros((V, r))
    W = np.zeros((V, r))
    d = oracle.draft_sample(U, E, W, [0], [1.0])
    assert d["lse"][0, 0] == pytest.approx(2.5 + math.log(V), abs=1e-12)
    assert d["logq"][0, 0] == pytest.approx(-math.log(V), abs=1e-12)


def test_single_spike_dominates_at_low_temperature():
    V, r = 512, 4
    U = np.zeros((3, 1, V))
    for b, spike in enumerate((7, 300, 511)):
        U[b, 0, spike] = 5.0
    d = oracle.draft_sample(U, np.zeros((V, r)), np.zeros((V, r)), [0, 0, 0], [0.05, 0.05, 0.05])
    assert list(d["tokens"][:, 0]) == [7, 300, 511]
    # logq = -log(1 + (V-1) exp(-100)) ~ 0
    assert np.all(np.abs(d["logq"]) < 1e-30)


def test_greedy_ties_take_lowest_id():
    V, r = 64, 4
    U = np.zeros((1, 2, V))
    U[0, 0, [5, 9, 40]] = 3.0
    U[0, 1, [63, 2]] = 1.0
    d = oracle.draft_sample(U, np.zeros((V, r)), np.zeros((V, r)), [1], [0.0])
    assert list(d["tokens"][0]) == [5, 2]
    assert d["lse"][0, 0] == 3.0 and d["logq"][0, 0] == 0.0
    assert d["gap"][0, 0] == 0.0


def test_markov_logits_equal_library_matmul():
    # z = fp32(U + W_out @ E_in[prev]), prev = anchor then the drawn tokens
    rng = np.random.default_rng(3)
    B, G, V, r = 3, 4, 97, 8
    U = rng.normal(0, 2, (B, G, V))
    E = rng.normal(0, 0.3, (V, r))
    W = rng.normal(0, 0.3, (V, r))
    anchor = np.array([0, 50, 96])
    d = oracle.draft_sample(U, E, W, anchor, [1.0, 0.0, 0.7], seed=9, want_z=True)
    for b in range(B):
        prev = anchor[b]
        for j in range(G):
            want = (U[b, j] + np.matmul(W, E[prev])).astype(np.float32).astype(np.float64)
            np.testing.assert_allclose(d["z"][b, j], want, rtol=0, atol=1e-6)
            prev = d["tokens"][b, j]


def test_gumbel_max_matches_softmax_distribution():
    V, r, N, T = 8, 2, 1000000, 0.8
    rng = np.random.default_rng(4)
    row = rng.normal(0, 1.5, V)
    U = np.broadcast_to(row, (N, 1, V)).copy()
    d = oracle.draft_sample(U, np.zeros((V, r)), np.zeros((V, r)), np.zeros(N, np.int32),
                            np.full(N, T), rid=np.arange(N), seed=11)
    counts = np.bincount(d["tokens"][:, 0], minlength=V)
    ok, chi2 = _chi2_ok(counts, _softmax(row / T), N)
    assert ok, chi2
    # logq is the log-probability of the drawn token
    p = _softmax(row / T)
    np.testing.assert_allclose(d["logq"][:, 0], np.log(p[d["tokens"][:, 0]]), atol=1e-12)


def test_second_position_conditions_on_first_draw():
    V, r, N, T = 5, 3, 200000, 1.0
    rng = np.random.default_rng(5)
    row0 = rng.normal(0, 1, V)
    row1 = rng.normal(0, 1, V)
    E = rng.normal(0, 1.0, (V, r))
    W = rng.normal(0, 1.0, (V, r))
    U = np.empty((N, 2, V))
    U[:, 0] = row0
    U[:, 1] = row1
    anchor = np.full(N, 2, np.int32)
    d = oracle.draft_sample(U, E, W, anchor, np.full(N, T), rid=np.arange(N), seed=21)
    x0, x1 = d["tokens"][:, 0], d["tokens"][:, 1]
    ok, chi2 = _chi2_ok(np.bincount(x0, minlength=V), _softmax((row0 + W @ E[2]) / T), N)
    assert ok, chi2
    for a in range(V):
        sel = x0 == a
        if sel.sum() < 2000:
            continue
        want = _softmax((row1 + W @ E[a]) / T)
        ok, chi2 = _chi2_ok(np.bincount(x1[sel], minlength=V), want, sel.sum())
        assert ok, (a, chi2)


def test_request_id_and_seed_select_independent_streams():
    V, r = 256, 2
    U = np.zeros((2, 3, V))
    kw = dict(E_in=np.zeros((V, r)), W_out=np.zeros((V, r)), anchor=[0, 0], temp=[1.0, 1.0])
    a = oracle.draft_sample(U, rid=[5, 5], seed=1, **kw)["tokens"]
    b = oracle.draft_sample(U, rid=[5, 6], seed=1, **kw)["tokens"]
    c = oracle.draft_sample(U, rid=[5, 5], seed=2, **kw)["tokens"]
    assert np.array_equal(a[0], a[1]) and np.array_equal(a[0], b[0])
    assert not np.array_equal(b[0], b[1]) and not np.array_equal(a[0], c[0])


def test_constant_rows_draw_the_argmax_of_the_token_uniforms():
    # equal logits: s_v + g(u_v) orders tokens as u_v does (g is increasing),
    # so the drawn token is the argmax of the token uniforms, each taken from
    # its own word (token slot v), the lowest id on an exact tie
    V, r, G = 64, 2, 3
    U = np.full((5, G, V), -1.25)
    rid = np.array([0, 3, 17, 1000, 77777], np.uint32)
    for seed in (0, 9, 123456789):
        d = oracle.draft_sample(U, np.zeros((V, r)), np.zeros((V, r)), np.zeros(5, np.int32),
                                np.full(5, 0.6), rid=rid, seed=seed)
        for b in range(5):
            for j in range(G):
                u = oracle.uniforms(seed, int(rid[b]), j, 0, V, 0)
                assert d["tokens"][b, j] == int(np.argmax(u))
                assert d["logq"][b, j] == pytest.approx(-math.log(V), abs=1e-12)


def test_two_token_row_accepts_the_larger_perturbed_logit():
    # V = 8 with only tokens 2 and 5 alive: token 5 wins exactly when
    # s5 - s2 > g(u2) - g(u5), i.e. when u5^exp(-s5) > u2^exp(-s2) (the
    # exponential-race form of the same comparison)
    V, r, N = 8, 2, 4000
    U = np.full((N, 1, V), -3.0e4)
    U[:, 0, 2] = 0.3
    U[:, 0, 5] = -0.4
    rid = np.arange(N, dtype=np.uint32)
    d = oracle.draft_sample(U, np.zeros((V, r)), np.zeros((V, r)), np.zeros(N, np.int32),
                            np.ones(N), rid=rid, seed=77)
    u2 = np.array([oracle.uniform(77, b, 0, 2, 0) for b in range(N)])
    u5 = np.array([oracle.uniform(77, b, 0, 5, 0) for b in range(N)])
    want = np.where(np.log(u5) * math.exp(0.4) > np.log(u2) * math.exp(-0.3), 5, 2)
    assert np.array_equal(d["tokens"][:, 0], want)
    p5 = math.exp(-0.4) / (math.exp(-0.4) + math.exp(0.3))
    assert abs((want == 5).mean() - p5) < 4 * math.sqrt(p5 * (1 - p5) / N)


def test_gumbel_max_matches_softmax_on_a_wider_row():
    V, r, N, T = 40, 2, 400000, 0.7
    rng = np.random.default_rng(14)
    row = rng.normal(0, 1.2, V)
    U = np.broadcast_to(row, (N, 1, V)).copy()
    d = oracle.draft_sample(U, np.zeros((V, r)), np.zeros((V, r)), np.zeros(N, np.int32),
                            np.full(N, T), rid=np.arange(N), seed=41)
    p = _softmax(row / T)
    ok, chi2 = _chi2_ok(np.bincount(d["tokens"][:, 0], minlength=V), p, N)
    assert ok, chi2
    # the reported gap is the distance between the two largest keys
    assert np.all(d["gap"][:, 0] >= 0) and np.all(np.isfinite(d["top"][:, 0]))


def test_masked_tokens_are_never_drawn_and_leave_lse_unchanged():
    """A masked token (logit -3e4) has probability exp(-3e4 / T) = 0 in double
    precision: the draft never draws it and lse is the log-sum-exp over the
    unmasked tokens alone, also for rows whose first tokens are all masked."""
    V, r, B, G = 96, 4, 6, 2
    rng = np.random.default_rng(3)
    U = rng.normal(0, 2, (B, G, V))
    mask = np.zeros(V, bool)
    mask[:40] = True          # the first 40 tokens
    mask[-12:] = True
    U[..., mask] = -3.0e4
    E = rng.normal(0, 0.3, (V, r))
    W = rng.normal(0, 0.3, (V, r))
    anchor = np.array([50, 60, 41, 77, 3, 95], np.int32)
    temps = np.array([1.0, 0.7, 1.3, 0.0, 1.0, 2.0])
    d = oracle.draft_sample(U, E, W, anchor, temps, seed=11)
    assert not mask[d["tokens"]].any()
    for b in range(B):
        prev = anchor[b]
        for j in range(G):
            z = (U[b, j] + W @ E[prev]).astype(np.float32).astype(np.float64)  # fp32 logits, as drawn
            zu = z[~mask]
            if temps[b] > 0:
                s = zu / temps[b]
                want = s.max() + math.log(np.exp(s - s.max()).sum())
            else:
                want = zu.max()
            assert d["lse"][b, j] == pytest.approx(want, rel=1e-12, abs=1e-9)
            prev = d["tokens"][b, j]
