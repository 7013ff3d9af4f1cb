"""Full-size draft logits against a plain PyTorch reference, and repeatability.

The draft kernels keep every logit on chip; asked to store them they also
write z = U_j + E_in[x_{j-1}] W_out^T, so every row, position and vocabulary
entry of a full-size batch can be checked against a float64 PyTorch matmul
(the oracle is too slow for that).  Repeated calls on the same inputs must
agree bit for bit: every random number comes from a counter-based Philox
stream and the partial states are merged in a fixed order, so any difference
between calls is a race in the kernels.
"""
import pytest
import torch

from speculative_decoding_draft_head_gb300 import binding
from speculative_decoding_draft_head_gb300.synth import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

FULL = ["qwen3", "dspark5", "largev", "highconc"]


def _draft(inp, seed, store_logits=False):
    return binding.draft_sample(inp["base"], inp["e_in"], inp["w_out"], inp["anchor"],
                                inp["temperature"], inp["request_id"], seed,
                                store_logits=store_logits)


@pytest.mark.parametrize("name", FULL)
def test_full_size_logits_match_torch(name):
    w = WORKLOADS[name]
    inp = make_inputs(w, 21, device="cuda")
    d = _draft(inp, 21, store_logits=True)
    torch.cuda.synchronize()
    tokens = d["tokens"]
    assert int((tokens < 0).sum()) == 0
    prev = torch.cat([inp["anchor"][:, None], tokens[:, :-1]], 1).long()
    e_in = inp["e_in"].double()
    w_out = inp["w_out"].double()
    for j in range(w.G):
        ref = inp["base"][:, j].double() + e_in[prev[:, j]] @ w_out.T
        err = (d["logits"][:, j].double() - ref).abs()
        # fp32 accumulation of exact bf16 products, then one fp32 add to U
        bad = err > 1e-5 + 1e-6 * ref.abs()
        assert not bool(bad.any()), "position %d: %d logits off, max error %.3g" % (
            j, int(bad.sum()), float(err.max()))
        del ref, err, bad


def _bits(t):
    if t.dtype in (torch.float32, torch.int32):
        return t.view(torch.int32)
    if t.dtype == torch.float64:
        return t.view(torch.int64)
    return t


@pytest.mark.parametrize("name", ["dspark5", "highconc", "largev"])
def test_repeated_calls_bitwise_identical(name):
    w = WORKLOADS[name]
    inp = make_inputs(w, 5, device="cuda")
    runs = []
    # the last call also stores the logits: a slower epilogue must not change anything
    for store in (False, False, True):
        d = _draft(inp, 5, store_logits=store)
        vl = None
        out = {"draft_" + k: v.clone() for k, v in d.items() if k != "logits"}
        if w.scheduler:
            s = binding.schedule_prefix(inp["conf_logits"], inp["pos_temp"], inp["sps"], w.L_min, w.G)
            vl = s["verify_len"]
            out.update({"sched_" + k: v.clone() for k, v in s.items()})
        v = binding.verify(inp["target"], inp["base"], inp["e_in"], inp["w_out"], inp["anchor"], d, vl,
                           inp["temperature"], inp["request_id"], 5)
        out.update({"verify_" + k: t.clone() for k, t in v.items()})
        torch.cuda.synchronize()
        runs.append(out)
    for i, r in enumerate(runs[1:], 1):
        for k, t in runs[0].items():
            same = torch.equal(_bits(t), _bits(r[k]))
            assert same, "call %d differs from call 0 in %s" % (i, k)
