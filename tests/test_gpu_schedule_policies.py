"""The scheduler's other verify-length policies on the GPU against the oracle.

Policies (see dspark_schedule_policy): best prefix without early stop (the
deployed mode, fed with confidences from two rounds back), and fixed
thresholds on the prefix survival a or on the per-position confidence c.
The scheduler is cheap, so the workloads run at full size, with the smooth
SPS table of the workloads and with a step-shaped one on which the best
prefix and the early stop differ.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_head_gb300 import binding
from speculative_decoding_draft_head_gb300.synth import WORKLOADS, make_inputs

from parity import REL, TIE_THETA

pytestmark = pytest.mark.gpu


def _step_sps(n, device):
    n_idx = torch.arange(n, dtype=torch.float64)
    table = torch.where(n_idx < 0.45 * n, 1.0, torch.where(n_idx < 0.7 * n, 0.75, 0.6))
    return table.to(torch.float32).to(device)


def _compare(g, o, threshold_policy):
    np.testing.assert_allclose(g["conf"].cpu().numpy(), o["conf"], rtol=REL, atol=0)
    np.testing.assert_allclose(g["cum_conf"].cpu().numpy(), o["cum_conf"], rtol=REL, atol=0)
    gl = g["verify_len"].cpu().numpy()
    near_tie = min(o["min_margin"], o["min_tie"]) <= (1e-5 if threshold_policy else TIE_THETA)
    if not np.array_equal(gl, o["verify_len"]):
        assert near_tie, "verify lengths differ in %d requests" % int((gl != o["verify_len"]).sum())
        return False
    theta = float(g["theta"].cpu().numpy()[0])
    assert abs(theta - o["theta"]) <= REL * max(1.0, abs(o["theta"]))
    return True


@pytest.mark.parametrize("name", ["dspark5", "highconc"])
@pytest.mark.parametrize("policy,threshold", [(binding.SCHED_BEST_PREFIX, 0.0),
                                              (binding.SCHED_THRESHOLD_CUM, 0.35),
                                              (binding.SCHED_THRESHOLD_CONF, 0.6)])
@pytest.mark.parametrize("table", ["smooth", "step"])
def test_policy_matches_oracle(name, policy, threshold, table):
    w = WORKLOADS[name]
    matched = 0
    for seed in range(4):
        inp = make_inputs(w, seed, device="cuda")
        sps = inp["sps"] if table == "smooth" else _step_sps(inp["sps"].numel(), "cuda")
        g = binding.schedule_prefix(inp["conf_logits"], inp["pos_temp"], sps, w.L_min, w.G,
                                    policy=policy, threshold=threshold)
        torch.cuda.synchronize()
        o = oracle.schedule_policy(inp["conf_logits"].cpu(), inp["pos_temp"].cpu(), sps.cpu(), w.L_min, w.G,
                                   policy, threshold)
        matched += _compare(g, o, policy >= binding.SCHED_THRESHOLD_CUM)
    assert matched >= 3


def test_best_prefix_differs_from_early_stop_on_a_step_table():
    w = WORKLOADS["dspark5"]
    inp = make_inputs(w, 1, device="cuda")
    sps = _step_sps(inp["sps"].numel(), "cuda")
    e = binding.schedule_prefix(inp["conf_logits"], inp["pos_temp"], sps, w.L_min, w.G)
    p = binding.schedule_prefix(inp["conf_logits"], inp["pos_temp"], sps, w.L_min, w.G,
                                policy=binding.SCHED_BEST_PREFIX)
    torch.cuda.synchronize()
    # the early stop halts at the first drop of the table; the best prefix may go past it
    assert float(p["theta"].cpu()[0]) >= float(e["theta"].cpu()[0]) * (1 - 1e-12)
    assert int(p["verify_len"].sum()) >= int(e["verify_len"].sum())


def test_unknown_policy_is_rejected():
    w = WORKLOADS["dspark5"].scaled(B=8)
    inp = make_inputs(w, 0, device="cuda")
    with pytest.raises(binding.DSparkError):
        binding.schedule_prefix(inp["conf_logits"], inp["pos_temp"], inp["sps"], w.L_min, w.G, policy=7)
    with pytest.raises(binding.DSparkError):
        binding.schedule_prefix(inp["conf_logits"], inp["pos_temp"], inp["sps"], w.L_min, w.G,
                                policy=binding.SCHED_THRESHOLD_CUM, threshold=float("nan"))


def test_lagged_scheduler_uses_the_confidences_of_two_rounds_back():
    # the deployed mode: round t is scheduled (best prefix, no early stop) from
    # round t - 2's calibrated confidences; the first two rounds use their own
    w = WORKLOADS["dspark5"]
    inp = make_inputs(w, 5, device="cuda")
    sched = binding.LaggedScheduler(inp["pos_temp"], inp["sps"], w.L_min, w.G, lag=2)
    gen = torch.Generator(device="cuda").manual_seed(5)
    rounds = [1.0 + torch.randn((w.B, w.G), generator=gen, device="cuda") for _ in range(5)]
    for t, cl in enumerate(rounds):
        g = sched.step(cl)
        torch.cuda.synchronize()
        src = rounds[t - 2] if t >= 2 else cl
        o = oracle.schedule_policy(src.cpu(), inp["pos_temp"].cpu(), inp["sps"].cpu(), w.L_min, w.G,
                                   binding.SCHED_BEST_PREFIX)
        _compare(g, o, False)
        if t >= 2:  # and not from its own round
            own = oracle.schedule_policy(cl.cpu(), inp["pos_temp"].cpu(), inp["sps"].cpu(), w.L_min, w.G,
                                         binding.SCHED_BEST_PREFIX)
            assert not np.array_equal(own["verify_len"], o["verify_len"])
