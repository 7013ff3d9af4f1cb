"""Pins for the oracle's rejection-sampling verification.

Sources: "Les mathematiques derriere l'acceleration" (seventnews.com),
sections "La garantie de l'echantillonnage par rejet" (accept with
min(1, p/q), stop at the first rejection, resample from the residual; output
identical in distribution to the target) and "Rendement attendu et formule
d'acceleration" (expected tokens per pass (1 - a^(g+1)) / (1 - a), about 2.8
at g = 4, a = 0.7); "DSpark, la bozza che sa quando fermarsi" (paithon.it),
section "Verificare meglio, non di piu'" (acceptance = 1 - TV(p, q));
"DeepSeek发布DSpark" (learnblockchain.cn), section "DSpark 是什么？" (bonus
token when the whole block is accepted).
"""
import itertools
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _softmax(x):
    e = np.exp(x - x.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def _chi2_ok(counts, probs, n, sigmas=6.0):
    exp = probs * n
    mask = exp > 0
    assert counts[~mask].sum() == 0, "mass on an impossible outcome"
    chi2 = (((counts - exp) ** 2)[mask] / exp[mask]).sum()
    dof = mask.sum() - 1
    return chi2 < dof + sigmas * math.sqrt(2 * dof), chi2


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(None, 1)
            vals[k] = v
    return vals


def _run(p_rows, q_rows, N, seed, temp=1.0, L=None):
    """Draft with q rows (no Markov bias) and verify against p rows, N requests."""
    G = len(q_rows)
    V = len(q_rows[0])
    r = 1
    U = np.broadcast_to(np.log(np.asarray(q_rows)) * temp, (N, G, V)).copy()
    tgt = np.broadcast_to(np.log(np.asarray(p_rows)) * temp, (N, G + 1, V)).copy()
    E = np.zeros((V, r))
    W = np.zeros((V, r))
    anchor = np.zeros(N, np.int32)
    temps = np.full(N, temp)
    rid = np.arange(N)
    d = oracle.draft_sample(U, E, W, anchor, temps, rid=rid, seed=seed)
    vl = None if L is None else np.full(N, L, np.int32)
    v = oracle.verify(tgt, U, E, W, anchor, d["tokens"], vl, temps, rid=rid, seed=seed)
    return d, v


def test_acceptance_probability_is_one_minus_tv():
    rng = np.random.default_rng(7)
    V, N = 8, 200000
    p = _softmax(rng.normal(0, 1.2, V))
    q = _softmax(rng.normal(0, 1.2, V))
    tv = 0.5 * np.abs(p - q).sum()
    alpha = np.minimum(p, q).sum()
    assert alpha == pytest.approx(1 - tv, abs=1e-15)
    d, v = _run([p, p], [q], N, seed=3, temp=1.3)
    acc = (v["accept_len"] >= 1).mean()
    assert abs(acc - alpha) < 4 * math.sqrt(alpha * (1 - alpha) / N), (acc, alpha)
    # the recorded acceptance threshold is min(1, p/q) of the drawn token
    x = d["tokens"][:, 0]
    # (the draft logits are held in fp32, so q carries a relative error of ~1e-7)
    np.testing.assert_allclose(np.exp(v["logp"][:, 0] - v["logq"][:, 0]), p[x] / q[x], rtol=2e-6)


def test_expected_tokens_per_pass_matches_closed_form_and_page_value():
    g = _read_golden("expected_tokens_per_pass.txt")
    gamma, alpha = int(g["gamma"]), float(g["alpha"])
    closed = (1 - alpha ** (gamma + 1)) / (1 - alpha)
    assert round(closed, int(g["printed_digits"])) == float(g["printed"])
    assert closed == pytest.approx(float(g["exact"]), abs=5e-6)
    # constructed rows: p uniform, q = p (1 +- 0.6) on the two halves -> sum min(p, q) = 0.7
    V, N = 10, 300000
    p = np.full(V, 1.0 / V)
    q = p * np.where(np.arange(V) < V // 2, 1.6, 0.4)
    assert np.minimum(p, q).sum() == pytest.approx(alpha, abs=1e-15)
    _, v = _run([p] * (gamma + 1), [q] * gamma, N, seed=5)
    mean = v["num_out"].mean()
    se = v["num_out"].std() / math.sqrt(N)
    assert abs(mean - closed) < 4 * se, (mean, closed, se)
    # every emitted sequence is the accepted prefix plus one token
    assert np.all(v["num_out"] == v["accept_len"] + 1)


def _exact_output_distribution(p0, p1, p2, q0, q1):
    """Exact law of the first three tokens (outputs continued with the target).

    p0[y0], p1[y0][y1], p2[y0][y1][y2]: target conditionals; q0[x0], q1[x0][x1]:
    draft conditionals (the second depends on the first draft token).
    """
    V = len(p0)
    out = np.zeros((V, V, V))

    def residual(p, q):
        res = np.maximum(p - q, 0.0)
        return res / res.sum() if res.sum() > 0 else p

    for x0 in range(V):
        if q0[x0] == 0:
            continue
        acc0 = min(1.0, p0[x0] / q0[x0])
        # rejection at position 0
        rej0 = q0[x0] * (1 - acc0)
        if rej0 > 0:
            r0 = residual(p0, q0)
            for y0, y1, y2 in itertools.product(range(V), repeat=3):
                out[y0, y1, y2] += rej0 * r0[y0] * p1[y0][y1] * p2[y0][y1][y2]
        for x1 in range(V):
            w = q0[x0] * acc0 * q1[x0][x1]
            if w == 0:
                continue
            acc1 = min(1.0, p1[x0][x1] / q1[x0][x1])
            r1 = residual(p1[x0], q1[x0])
            for y1, y2 in itertools.product(range(V), repeat=2):
                out[x0, y1, y2] += w * (1 - acc1) * r1[y1] * p2[x0][y1][y2]
            for y2 in range(V):
                out[x0, x1, y2] += w * acc1 * p2[x0][x1][y2]
    return out


def _toy_tables(seed, V=4):
    rng = np.random.default_rng(seed)
    p0 = _softmax(rng.normal(0, 1, V))
    p1 = _softmax(rng.normal(0, 1, (V, V)))
    p2 = _softmax(rng.normal(0, 1, (V, V, V)))
    q0 = _softmax(rng.normal(0, 1, V))
    q1 = _softmax(rng.normal(0, 1, (V, V)))
    return p0, p1, p2, q0, q1


def test_exact_enumeration_is_lossless():
    # the enumeration itself: its law of the first three tokens is the
    # target's joint (and the mirrored residual max(0, q - p) is not)
    for seed in range(5):
        p0, p1, p2, q0, q1 = _toy_tables(seed)
        got = _exact_output_distribution(p0, p1, p2, q0, q1)
        want = p0[:, None, None] * p1[:, :, None] * p2
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)
    p0, p1, p2, q0, q1 = _toy_tables(0)
    swapped = _exact_output_distribution(q0, q1, p2, p0, p1)
    assert np.abs(swapped - (p0[:, None, None] * p1[:, :, None] * p2)).max() > 1e-3


def _continue_with_target(out, n_out, p1, p2, rng):
    """Extend each emitted sequence to three tokens with the target's own
    conditionals (inverse CDF on seeded uniforms)."""
    N = len(n_out)
    y = out[:, :3].copy()
    u = rng.random((N, 2))
    short1 = n_out < 2
    c1 = np.cumsum(p1[y[:, 0]], axis=1)
    y[short1, 1] = np.minimum((c1[short1] <= u[short1, :1]).sum(axis=1), p1.shape[1] - 1)
    short2 = n_out < 3
    c2 = np.cumsum(p2[y[:, 0], y[:, 1]], axis=1)
    y[short2, 2] = np.minimum((c2[short2] <= u[short2, 1:]).sum(axis=1), p2.shape[2] - 1)
    return y


def test_brute_force_enumeration_matches_the_oracle_end_to_end():
    """V = 4, gamma = 2, 10^6 rounds through the oracle's draft and verify.

    The draft is a Markov head (position 1 depends on the first draft token) and
    the target rows depend on the drafted prefix.  Brute-force enumeration of
    every draft path, accept path and residual / bonus outcome, with the
    probabilities the oracle itself reports (its log q of each drafted token,
    its log p of each tested one), gives the exact law of the first three
    tokens (short outputs continued with the target's conditionals); the
    oracle's empirical law over 10^6 seeded rounds must match it by
    chi-square on the first token, the first two and all three, and the
    enumeration must equal the target's joint."""
    V, N, T, seed = 4, 1000000, 1.0, 17
    p0, p1, p2, q0, q1 = _toy_tables(11, V)
    # draft: U row 0 = log q0 (the anchor's bias removed); row 1 = 0 plus the
    # bias W_out @ E_in[x0] = log q1[x0]
    r = V
    E = np.eye(V)
    W = np.log(q1).T          # W_out[v, k] = log q1[k][v]
    U = np.zeros((N, 2, V))
    U[:, 0] = np.log(q0) - (W @ E[0])      # position 0 is biased by the anchor (token 0)
    anchor = np.zeros(N, np.int32)
    temps = np.full(N, T)
    rid = np.arange(N)
    d = oracle.draft_sample(U, E, W, anchor, temps, rid=rid, seed=seed)
    x = d["tokens"]
    tgt = np.empty((N, 3, V))
    tgt[:, 0] = np.log(p0)
    tgt[:, 1] = np.log(p1[x[:, 0]])
    tgt[:, 2] = np.log(p2[x[:, 0], x[:, 1]])
    v = oracle.verify(tgt, U, E, W, anchor, x, None, temps, rid=rid, seed=seed)
    # the draft and target probabilities the oracle used, per path: its drafted
    # log q and tested log p, gathered back into tables for the enumeration
    q0_or = np.full(V, np.nan)
    q1_or = np.full((V, V), np.nan)
    p0_or = np.full(V, np.nan)
    p1_or = np.full((V, V), np.nan)
    q0_or[x[:, 0]] = np.exp(d["logq"][:, 0])
    q1_or[x[:, 0], x[:, 1]] = np.exp(d["logq"][:, 1])
    p0_or[x[:, 0]] = np.exp(v["logp"][:, 0])
    t1 = ~np.isnan(v["logp"][:, 1])
    p1_or[x[t1, 0], x[t1, 1]] = np.exp(v["logp"][t1, 1])
    assert not np.isnan(q0_or).any() and not np.isnan(q1_or).any()
    assert not np.isnan(p0_or).any() and not np.isnan(p1_or).any()
    # (z is held in fp32, so the oracle's q carries a relative error of ~1e-7)
    np.testing.assert_allclose(q0_or, q0, rtol=1e-6)
    np.testing.assert_allclose(q1_or, q1, rtol=1e-6)
    np.testing.assert_allclose(p0_or, p0, rtol=1e-12)
    np.testing.assert_allclose(p1_or, p1, rtol=1e-12)
    exact = _exact_output_distribution(p0_or, p1_or, p2, q0_or, q1_or)
    np.testing.assert_allclose(exact, p0[:, None, None] * p1[:, :, None] * p2, rtol=0, atol=1e-6)
    y = _continue_with_target(v["out_tokens"], v["num_out"], p1, p2, np.random.default_rng(99))
    ok, chi2 = _chi2_ok(np.bincount(y[:, 0], minlength=V), exact.sum(axis=(1, 2)), N)
    assert ok, chi2
    ok, chi2 = _chi2_ok(np.bincount(y[:, 0] * V + y[:, 1], minlength=V * V), exact.sum(axis=2).ravel(), N)
    assert ok, chi2
    ok, chi2 = _chi2_ok(np.bincount((y[:, 0] * V + y[:, 1]) * V + y[:, 2], minlength=V ** 3), exact.ravel(), N)
    assert ok, chi2
    # the paths are all exercised: rejections at 0 and 1, full acceptances
    k = v["accept_len"]
    assert min((k == 0).mean(), (k == 1).mean(), (k == 2).mean()) > 0.05
    # the draft second position really depends on the first (the Markov head)
    assert np.abs(q1[0] - q1[1]).max() > 0.05


def test_a_lossy_verifier_fails_the_end_to_end_law():
    """The chi-square above has the power to see a wrong residual: feeding the
    oracle's rejected rows a residual of max(0, q - p) (by swapping the roles
    of draft and target in the tables) moves the law far outside the bound."""
    V, N, seed = 4, 200000, 3
    p0, p1, p2, q0, q1 = _toy_tables(11, V)
    wrong = _exact_output_distribution(q0, q1, p2, p0, p1)
    right = p0[:, None, None] * p1[:, :, None] * p2
    rng = np.random.default_rng(seed)
    sample = rng.choice(V ** 3, size=N, p=wrong.ravel() / wrong.sum())
    ok, _ = _chi2_ok(np.bincount(sample, minlength=V ** 3), right.ravel(), N)
    assert not ok


def test_greedy_limit_is_argmax_prefix_match():
    V, G, r = 16, 4, 2
    U = np.zeros((3, G, V))
    # draft greedy tokens 3, 5, 7, 9
    for j, tok in enumerate((3, 5, 7, 9)):
        U[:, j, tok] = 1.0
    tgt = np.zeros((3, G + 1, V))
    # request 0: target agrees on 0, 1, disagrees at 2 (argmax 11)
    for j, tok in enumerate((3, 5, 11, 9, 2)):
        tgt[0, j, tok] = 2.0
    # request 1: agrees everywhere; bonus from row 4 (argmax 13, tie with 14 -> 13)
    for j, tok in enumerate((3, 5, 7, 9, 13)):
        tgt[1, j, tok] = 2.0
    tgt[1, 4, 14] = 2.0
    # request 2: verify length 2; bonus from row 2 (argmax 6)
    for j, tok in enumerate((3, 5, 6, 0, 0)):
        tgt[2, j, tok] = 2.0
    E, W = np.zeros((V, r)), np.zeros((V, r))
    anchor = np.zeros(3, np.int32)
    temps = np.zeros(3)
    d = oracle.draft_sample(U, E, W, anchor, temps)
    assert d["tokens"].tolist() == [[3, 5, 7, 9]] * 3
    v = oracle.verify(tgt, U, E, W, anchor, d["tokens"], np.array([4, 4, 2], np.int32), temps)
    assert v["accept_len"].tolist() == [2, 4, 2]
    assert v["out_tokens"][0].tolist() == [3, 5, 11, -1, -1]
    assert v["out_tokens"][1].tolist() == [3, 5, 7, 9, 13]
    assert v["out_tokens"][2].tolist() == [3, 5, 6, -1, -1]
    assert v["num_out"].tolist() == [3, 5, 3]
    assert v["final_kind"].tolist() == [3, 0, 0]


def test_verify_length_zero_emits_one_target_token():
    V, G, r, N = 6, 3, 1, 100000
    rng = np.random.default_rng(8)
    p = _softmax(rng.normal(0, 1, V))
    U = np.zeros((N, G, V))
    tgt = np.broadcast_to(np.log(p), (N, G + 1, V)).copy()
    E, W = np.zeros((V, r)), np.zeros((V, r))
    anchor = np.zeros(N, np.int32)
    temps = np.ones(N)
    d = oracle.draft_sample(U, E, W, anchor, temps, rid=np.arange(N), seed=2)
    v = oracle.verify(tgt, U, E, W, anchor, d["tokens"], np.zeros(N, np.int32), temps,
                      rid=np.arange(N), seed=2)
    assert np.all(v["accept_len"] == 0) and np.all(v["num_out"] == 1)
    ok, chi2 = _chi2_ok(np.bincount(v["out_tokens"][:, 0], minlength=V), p, N)
    assert ok, chi2


def test_markov_head_fixes_the_multimodal_collision():
    """'of course' / 'no problem': tokens of=0, course=1, no=2, problem=3."""
    V, N, big = 4, 40000, 40.0
    p0 = np.array([0.0, -big, 0.0, -big])
    p1 = {0: np.array([-big, 0.0, -big, -big]), 2: np.array([-big, -big, -big, 0.0])}
    results = {}
    for head in ("parallel", "markov"):
        r = V
        E = np.eye(V)
        W = np.zeros((V, r))
        if head == "markov":
            W[:, 0] = [0.0, big / 2, 0.0, -big / 2]
            W[:, 2] = [0.0, -big / 2, 0.0, big / 2]
        U = np.zeros((N, 2, V))
        U[:, 0] = p0
        U[:, 1] = [-big, 0.0, -big, 0.0]
        anchor = np.full(N, 1, np.int32)     # the anchor token adds no bias (W[:, 1] = 0)
        temps = np.ones(N)
        rid = np.arange(N)
        d = oracle.draft_sample(U, E, W, anchor, temps, rid=rid, seed=4)
        x0 = d["tokens"][:, 0]
        tgt = np.zeros((N, 3, V))
        tgt[:, 0] = p0
        tgt[:, 1] = np.where((x0 == 0)[:, None], p1[0], p1[2])
        v = oracle.verify(tgt, U, E, W, anchor, d["tokens"], None, temps, rid=rid, seed=4)
        first = v["accept_len"] >= 1
        assert first.all()
        results[head] = (v["accept_len"] == 2).mean()
    assert abs(results["parallel"] - 0.5) < 4 * math.sqrt(0.25 / N)
    assert results["markov"] == 1.0


def test_residual_and_bonus_draws_follow_their_laws():
    """One draft position (L = 1) on a 40-token vocabulary: the first emitted
    token is the accepted draft token or the residual draw and must have law
    p0; on a rejection it must have the residual law normalise(max(0, p0 - q0));
    when the draft token is accepted, the second emitted token is the bonus
    draw from p1.  Both are per-token Gumbel-max draws (streams 2 and 3)."""
    V, N, seed = 40, 1000000, 23
    rng = np.random.default_rng(31)
    p0 = _softmax(rng.normal(0, 1.0, V))
    q0 = _softmax(rng.normal(0, 1.0, V))
    p1 = _softmax(rng.normal(0, 1.5, V))
    d, v = _run([p0, p1], [q0], N, seed, L=1)
    first = v["out_tokens"][:, 0]
    ok, chi2 = _chi2_ok(np.bincount(first, minlength=V), p0, N)
    assert ok, chi2
    resid = np.maximum(p0 - q0, 0)
    assert (resid > 0).sum() > 10
    acc = v["accept_len"] == 1
    assert 0.3 < acc.mean() < 0.9
    ok, chi2 = _chi2_ok(np.bincount(v["out_tokens"][acc, 1], minlength=V), p1, int(acc.sum()))
    assert ok, chi2
    rej = ~acc
    ok, chi2 = _chi2_ok(np.bincount(first[rej], minlength=V), resid / resid.sum(), int(rej.sum()))
    assert ok, chi2
    assert np.all(v["final_kind"][rej] == 1) and np.all(v["final_kind"][acc] == 0)
    assert np.all(v["final_gap"] >= 0)


def test_target_masked_tokens_are_rejected_and_never_emitted():
    """Tokens the target masks (logit -3e4, probability 0) are rejected when
    drafted (p = 0 < u q) and never emitted by the residual or bonus draw."""
    V, G, r, B = 64, 3, 2, 400
    rng = np.random.default_rng(21)
    U = rng.normal(0, 1.5, (B, G, V))
    tgt = np.concatenate([U, rng.normal(0, 1.5, (B, 1, V))], axis=1) + rng.normal(0, 0.5, (B, G + 1, V))
    banned = np.zeros(V, bool)
    banned[rng.choice(V, 20, replace=False)] = True
    tgt[..., banned] = -3.0e4
    E, W = rng.normal(0, 0.2, (V, r)), rng.normal(0, 0.2, (V, r))
    anchor = rng.integers(0, V, B).astype(np.int32)
    temps = np.where(np.arange(B) % 4 == 0, 0.0, 1.0)
    d = oracle.draft_sample(U, E, W, anchor, temps, rid=np.arange(B), seed=5)
    v = oracle.verify(tgt, U, E, W, anchor, d["tokens"], None, temps, rid=np.arange(B), seed=5)
    drafted_banned = 0
    for b in range(B):
        k = v["accept_len"][b]
        out = v["out_tokens"][b, : v["num_out"][b]]
        assert not banned[out].any()
        # the first drafted banned token is never accepted
        hit = np.flatnonzero(banned[d["tokens"][b]])
        if hit.size:
            drafted_banned += 1
            assert k <= hit[0]
    assert drafted_banned > 20  # the case is exercised
