"""The recurrent (RNN) draft head on the GPU against the oracle, through the C ABI.

The head is the Markov head with its bias driven by a state
h_j = bf16(tanh(E_in[x_{j-1}] + W_h h_{j-1})) ("DSpark, la bozza che sa quando
fermarsi", section "Un po' di autoregressione basta", with the cell of the
oracle's reading).  Compared element by element: the drawn tokens (bit-exact
outside the oracle's near-ties), lse and log q (REL), the bf16 states
(bit-exact outside a rounding boundary closer than H_TIE), the stored logits,
and the verification of the drafted block through the stored logits.  A
mismatching token ends the comparison of its request (later positions see
another prefix).
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_head_gb300 import binding
from speculative_decoding_draft_head_gb300.synth import WORKLOADS, make_inputs, make_rnn_head

from parity import REL, Tally, compare_draft, compare_verify

pytestmark = pytest.mark.gpu

# the device state sum is compensated and tanh is taken in fp64: a state may
# differ from the oracle's only this close (relative) to a bf16 rounding boundary
H_TIE = 1e-12

SMALL = {
    # two row tiles with a ragged tail, a vocabulary of 32 tiles plus 8, T ~ U[0.3, 1.2]
    "ragged": WORKLOADS["highconc"].scaled(B=150, G=4, V=4104, r=64),
    # full rank, half the requests greedy
    "greedy_mix": WORKLOADS["largev"].scaled(B=40, G=6, V=2056, r=256),
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    binding.load()
    oracle.build()


def _gpu_draft(inp, head, seed):
    d = binding.draft_sample_rnn(inp["base"], head["e_in"], head["w_h"], head["w_out"], inp["anchor"],
                                 inp["temperature"], inp["request_id"], seed, store_logits=True,
                                 store_states=True)
    torch.cuda.synchronize()
    return d


def _oracle_draft(inp, head, seed, reqs):
    rid = inp["request_id"].cpu().numpy().astype(np.uint32)[reqs]
    return oracle.draft_sample_rnn_parallel(inp["base"].cpu()[reqs], head["e_in"].cpu(), head["w_h"].cpu(),
                                            head["w_out"].cpu(), inp["anchor"].cpu()[reqs],
                                            inp["temperature"].cpu()[reqs], rid, seed, want_z=True)


def _compare_states_and_logits(g, o, reqs, tally):
    gh = g["h"].float().cpu().numpy()
    gz = g["logits"].cpu().numpy()
    gt = g["tokens"].cpu().numpy()
    G = o["tokens"].shape[1]
    for i, b in enumerate(reqs):
        for j in range(G):
            # h_j and z_j depend on x_0 .. x_{j-1}: compare while those agree
            if j > 0 and gt[b, j - 1] != o["tokens"][i, j - 1]:
                break
            tally.decisions += 1
            if not np.array_equal(gh[b, j], o["h"][i, j]):
                if o["h_margin"][i, j] <= H_TIE:
                    tally.exempt += 1
                    break
                k = int(np.argmax(gh[b, j] != o["h"][i, j]))
                tally.failures.append("state b=%d j=%d unit %d gpu=%r oracle=%r margin=%.3g" %
                                      (b, j, k, gh[b, j, k], o["h"][i, j, k], o["h_margin"][i, j]))
                break
            err = np.abs(gz[b, j] - o["z"][i, j]) / np.maximum(1.0, np.abs(o["z"][i, j]))
            if err.max() > REL:
                tally.failures.append("logits b=%d j=%d max rel err %.3g" % (b, j, err.max()))


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("seed", [0, 1])
def test_small_workload_matches_oracle(name, seed):
    w = SMALL[name]
    inp = make_inputs(w, seed, device="cuda")
    head = make_rnn_head(w, seed, device="cuda")
    g = _gpu_draft(inp, head, seed)
    reqs = np.arange(w.B)
    o = _oracle_draft(inp, head, seed, reqs)
    gh = {k: v.cpu() for k, v in g.items()}
    t, _ = compare_draft(gh, o, inp["temperature"].cpu().numpy(), reqs)
    _compare_states_and_logits(g, o, reqs, t)
    t.check()
    assert t.exempt <= t.allowed_exempt()
    # the recurrence matters: states at j >= 1 differ from tanh(E_in[x_{j-1}])
    e = head["e_in"].float().cpu().numpy()
    prev = np.concatenate([inp["anchor"].cpu().numpy()[:, None], o["tokens"][:, :-1]], axis=1)
    assert np.mean(np.abs(o["h"][:, 1:] - np.tanh(e[prev[:, 1:]]))) > 1e-3


def test_full_size_sampled_requests():
    w = WORKLOADS["dspark5"]
    seed = 3
    inp = make_inputs(w, seed, device="cuda")
    head = make_rnn_head(w, seed, device="cuda")
    g = _gpu_draft(inp, head, seed)
    reqs = np.array([0, 1, 37, 100, 127, 128, 129, 200, 254, 255])
    o = _oracle_draft(inp, head, seed, reqs)
    gh = {k: v.cpu() for k, v in g.items()}
    t, _ = compare_draft(gh, o, inp["temperature"].cpu().numpy(), reqs)
    _compare_states_and_logits(g, o, reqs, t)
    t.check()
    # properties over every request: tokens in range, log q <= 0, |h| <= 1
    tok = g["tokens"].cpu().numpy()
    assert tok.min() >= 0 and tok.max() < w.V
    assert float(g["logq"].max()) <= 0.0
    assert float(g["h"].float().abs().max()) <= 1.0


@pytest.mark.parametrize("seed", [0, 5])
def test_verify_through_stored_logits(seed):
    w = SMALL["ragged"]
    inp = make_inputs(w, seed, device="cuda")
    head = make_rnn_head(w, seed, device="cuda")
    g = _gpu_draft(inp, head, seed)
    vl = torch.full((w.B,), w.G, dtype=torch.int32, device="cuda")
    vl[::3] = 1
    v = binding.verify(inp["target"], None, None, None, inp["anchor"], g, vl, inp["temperature"],
                       inp["request_id"], seed, draft_logits=g["logits"])
    torch.cuda.synchronize()
    reqs = np.arange(w.B)
    o = _oracle_draft(inp, head, seed, reqs)
    temps = inp["temperature"].cpu().numpy()
    t, diverged = compare_draft({k: x.cpu() for k, x in g.items()}, o, temps, reqs)
    # the oracle's verification with the head's own logits as the base and a
    # zero Markov bias: fp32(z + 0) = z, the recurrent head's draft distribution
    zeros = np.zeros((w.V, w.r))
    rid = inp["request_id"].cpu().numpy().astype(np.uint32)
    ov = oracle.verify_parallel(inp["target"].cpu(), o["z"], zeros, zeros, inp["anchor"].cpu(), o["tokens"],
                                vl.cpu().numpy(), temps, rid, seed)
    t.add(compare_verify({k: x.cpu() for k, x in v.items()}, ov, temps, reqs, diverged))
    t.check()
    assert t.exempt <= t.allowed_exempt()


def test_invalid_inputs():
    w = SMALL["ragged"].scaled(B=4)
    inp = make_inputs(w, 0, device="cuda")
    head = make_rnn_head(w, 0, device="cuda")
    anchor = inp["anchor"].clone()
    anchor[1] = -3
    ws = binding.default_workspace(binding.WS_DRAFT_RNN, w.B, w.G, w.V, w.r, anchor.device)
    d = binding.draft_sample_rnn(inp["base"], head["e_in"], head["w_h"], head["w_out"], anchor,
                                 inp["temperature"], None, 0, workspace=ws, store_states=True)
    assert binding.read_device_flags(ws) & binding.FLAG_BAD_TOKEN
    tok = d["tokens"].cpu().numpy()
    assert np.all(tok[1] == -1) and np.all(tok[[0, 2, 3]] >= 0)
    # fp32 weights are not supported by the recurrent head
    lib = binding.load()
    f = torch.zeros(16, device="cuda")
    st = lib.dspark_draft_sample_rnn(*([binding._ptr(f)] * 7), 1, 1, 8, 16, binding.DSPARK_F32, 0,
                                     *([binding._ptr(f)] * 5), binding._ptr(f), 1 << 20, None)
    assert st != 0 and b"bf16" in lib.dspark_last_error()
    # a workspace sized for the Markov head is too small (the states live there too)
    small = binding.default_workspace(binding.WS_DRAFT, w.B, w.G, w.V, w.r, anchor.device)
    with pytest.raises(binding.DSparkError):
        binding.draft_sample_rnn(inp["base"], head["e_in"], head["w_h"], head["w_out"], anchor,
                                 inp["temperature"], None, 0, workspace=small)
