"""Pins of the oracle's recurrent (RNN) draft head.

The pages name a recurrent head beside the Markov head ("DSpark, la bozza che
sa quando fermarsi", section "Un po' di autoregressione basta") without giving
its cell; the oracle reads it as h_j = bf16(tanh(E_in[x_{j-1}] + W_h h_{j-1}))
with h_{-1} = 0 and bias_j = h_j W_out^T.  Pins:
  - with W_h = 0 and the embedding table replaced by atanh(E_in), the state is
    exactly E_in[x_{j-1}] again, so the draft equals the (pinned) Markov head's;
  - the state carries the whole prefix: with W_h != 0 the logits of position 2
    change with x_0 even when x_1 is the same (the Markov head's do not);
  - in the linear regime (tiny weights) the states follow the linear recurrence
    e + W_h h within the bf16 rounding, which fixes the orientation of W_h;
  - every state is a bf16 value with |h| <= 1.
"""
import numpy as np
import pytest

import oracle


def _inputs(rng, B, G, V, r, wh_scale, e_scale=0.02):
    U = rng.normal(0, 2, (B, G, V))
    E = np.asarray(rng.normal(0, e_scale, (V, r)), np.float32).astype(np.float64)
    W = np.asarray(rng.normal(0, 0.02, (V, r)), np.float32).astype(np.float64)
    Wh = np.asarray(rng.normal(0, wh_scale, (r, r)), np.float32).astype(np.float64)
    anchor = rng.integers(0, V, B).astype(np.int32)
    return U, E, W, Wh, anchor


def _bf16(x):
    return (np.asarray(x, np.float32).view(np.uint32) & 0xFFFF0000).view(np.float32)


def test_zero_recurrence_with_atanh_table_is_the_markov_head():
    rng = np.random.default_rng(21)
    B, G, V, r = 6, 4, 64, 16
    U, E, W, _, anchor = _inputs(rng, B, G, V, r, 0.0)
    E = _bf16(E).astype(np.float64)          # bf16 values, as the head stores them
    temp = np.array([1.0, 0.7, 1.3, 0.0, 1.0, 0.5])
    m = oracle.draft_sample(U, E, W, anchor, temp, seed=5, want_z=True)
    n = oracle.draft_sample_rnn(U, np.arctanh(E), np.zeros((r, r)), W, anchor, temp, seed=5, want_z=True)
    assert np.array_equal(m["tokens"], n["tokens"])
    np.testing.assert_allclose(n["z"], m["z"], rtol=0, atol=0)
    np.testing.assert_allclose(n["lse"], m["lse"], rtol=1e-15)
    prev = np.concatenate([anchor[:, None], m["tokens"][:, :-1]], axis=1)
    np.testing.assert_array_equal(n["h"], E[prev])


def test_state_carries_the_whole_prefix():
    rng = np.random.default_rng(22)
    V, r = 32, 16
    U, E, W, Wh, _ = _inputs(rng, 1, 3, V, r, 0.3, e_scale=0.3)
    U[:] = -50.0
    # force x_0 then x_1 = 7 by huge base logits at positions 0 and 1
    outs = []
    for x0 in (3, 11):
        Uc = U.copy()
        Uc[0, 0, x0] = 50.0
        Uc[0, 1, 7] = 50.0
        d = oracle.draft_sample_rnn(Uc, E, Wh, W, np.array([0], np.int32), np.array([1.0]), seed=1, want_z=True)
        assert d["tokens"][0, :2].tolist() == [x0, 7]
        outs.append(d)
    # same x_1, different x_0: position 2 sees a different state and bias
    assert not np.array_equal(outs[0]["h"][0, 2], outs[1]["h"][0, 2])
    assert np.max(np.abs(outs[0]["z"][0, 2] - outs[1]["z"][0, 2])) > 1e-4
    # the Markov head conditions on x_1 only
    mk = [oracle.draft_sample(np.where(np.arange(V) == x0, 50.0, -50.0)[None, None, :].repeat(3, 1)
                              * np.array([1, 0, 0])[None, :, None] + np.where(np.arange(V) == 7, 50.0, -50.0)
                              [None, None, :] * np.array([0, 1, 0])[None, :, None] + U * np.array([0, 0, 1])[None, :, None],
                              E, W, np.array([0], np.int32), np.array([1.0]), seed=1, want_z=True)
          for x0 in (3, 11)]
    np.testing.assert_array_equal(mk[0]["z"][0, 2], mk[1]["z"][0, 2])


def test_linear_regime_follows_the_linear_recurrence():
    rng = np.random.default_rng(23)
    B, G, V, r = 3, 4, 40, 16
    U, E, W, Wh, anchor = _inputs(rng, B, G, V, r, 0.2, e_scale=1e-3)
    Wh = Wh * np.triu(np.ones((r, r)))      # not symmetric: fixes the orientation
    d = oracle.draft_sample_rnn(U, E, Wh, W, anchor, np.ones(B), seed=3)
    prev = np.concatenate([anchor[:, None], d["tokens"][:, :-1]], axis=1)
    for b in range(B):
        h = np.zeros(r)
        for j in range(G):
            lin = E[prev[b, j]] + Wh @ h
            np.testing.assert_allclose(d["h"][b, j], lin, rtol=2e-2, atol=1e-9)
            h = d["h"][b, j]
    # the transposed recurrence is not what the oracle computes
    h1 = d["h"][0, 0]
    lin1_t = E[prev[0, 1]] + Wh.T @ h1
    assert not np.allclose(d["h"][0, 1], lin1_t, rtol=2e-2, atol=1e-9)


def test_states_are_bounded_bf16_values():
    rng = np.random.default_rng(24)
    U, E, W, Wh, anchor = _inputs(rng, 4, 5, 48, 32, 0.5, e_scale=1.0)
    d = oracle.draft_sample_rnn(U, E, Wh, W, anchor, np.ones(4), seed=9)
    h = d["h"]
    assert np.all(np.abs(h) <= 1.0)
    np.testing.assert_array_equal(_bf16(h).astype(np.float64), h)
    assert np.all(d["h_margin"] >= 0)
