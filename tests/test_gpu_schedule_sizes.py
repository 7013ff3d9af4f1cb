"""The prefix scheduler against the oracle at candidate counts that reach
every form of its sort: one key per thread (up to 1024 candidates, including
counts that are not powers of two and a single candidate), two, four and eight
keys per thread in registers, and the shared-memory network beyond 8192
candidates, up to the largest batch the entry point takes (B * G = 16384).

A step-shaped SPS table puts the early stop at a chosen share of the
candidates, so the sorted order decides which requests gain a position at
that cut ("DSpark, la bozza che sa quando fermarsi", section "Verificare
meglio, non di piu'": candidates are admitted in decreasing a while
Theta = tau * SPS grows).
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_head_gb300 import binding
from speculative_decoding_draft_head_gb300.synth import WORKLOADS, make_inputs

from parity import REL, TIE_THETA

pytestmark = pytest.mark.gpu

# (B, G, L_min, L_max): candidates B * (L_max - L_min)
SIZES = [
    (1, 1, 0, 1),       # 1
    (3, 5, 1, 5),       # 12
    (31, 2, 1, 2),      # 31
    (33, 4, 1, 4),      # 99
    (256, 5, 1, 5),     # 1024
    (300, 5, 1, 5),     # 1200: two keys per thread
    (400, 6, 1, 6),     # 2000
    (1024, 4, 1, 4),    # 3072: four keys per thread
    (700, 8, 1, 8),     # 4900: eight keys per thread
    (1100, 9, 2, 9),    # 7700
    (1000, 10, 1, 9),   # 8000, L_max < G
    (4096, 4, 1, 4),    # 12288: shared-memory sort
    (2048, 8, 0, 8),    # 16384
]


def _step_table(B, L_min, ncand, share, n, device):
    """SPS(k) = 1 up to the cut B (L_min + 1) + share * ncand, 0.5 after."""
    cut = B * (L_min + 1) + int(share * ncand)
    k = torch.arange(n, dtype=torch.float64)
    return torch.where(k <= cut, 1.0, 0.5).to(torch.float32).to(device)


def _check(g, o):
    np.testing.assert_allclose(g["conf"].cpu().numpy(), o["conf"], rtol=REL, atol=0)
    np.testing.assert_allclose(g["cum_conf"].cpu().numpy(), o["cum_conf"], rtol=REL, atol=0)
    gl = g["verify_len"].cpu().numpy()
    if not np.array_equal(gl, o["verify_len"]):
        assert min(o["min_margin"], o["min_tie"]) <= TIE_THETA, \
            "verify lengths differ in %d requests" % int((gl != o["verify_len"]).sum())
        return False
    theta = float(g["theta"].cpu().numpy()[0])
    assert abs(theta - o["theta"]) <= REL * max(1.0, abs(o["theta"]))
    return True


@pytest.mark.parametrize("B,G,L_min,L_max", SIZES)
def test_schedule_matches_oracle_at_every_sort_size(B, G, L_min, L_max):
    w = WORKLOADS["dspark5"].scaled(B=B, G=G, V=16, r=16, L_min=L_min)
    ncand = B * (L_max - L_min)
    matched = total = 0
    for seed in range(2):
        inp = make_inputs(w, seed, device="cuda")
        n = B * (L_max + 1) + 1
        tables = [(None, inp["sps"][:n].contiguous())]
        tables += [(share, _step_table(B, L_min, ncand, share, n, "cuda")) for share in (0.3, 0.8)]
        for share, sps in tables:
            for policy in (binding.SCHED_EARLY_STOP, binding.SCHED_BEST_PREFIX):
                g = binding.schedule_prefix(inp["conf_logits"], inp["pos_temp"], sps, L_min, L_max,
                                            policy=policy)
                torch.cuda.synchronize()
                o = oracle.schedule_policy(inp["conf_logits"].cpu(), inp["pos_temp"].cpu(), sps.cpu(),
                                           L_min, L_max, policy)
                total += 1
                matched += _check(g, o)
                if share is not None and policy == binding.SCHED_EARLY_STOP:
                    # the early stop admits exactly the candidates before the cut
                    assert int(o["verify_len"].sum()) == B * L_min + int(share * ncand)
    # every mismatch is an oracle-marked near-tie (checked above); they stay rare
    assert matched >= total * 3 // 4
