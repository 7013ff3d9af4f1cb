"""Failure detection on the GPU without a fault.

Every wait in the library's kernels (mbarrier phases, the grid barrier between
block positions) is bounded: after its limit the kernel raises the timeout
flag and returns instead of spinning.  dspark_selftest_bounded_wait runs the
same wait helpers on an mbarrier phase and a counter that nothing completes,
with a short limit; both must give up and report it, and the context must stay
usable for ordinary calls.
"""
import time

import numpy as np
import pytest
import torch

from speculative_decoding_draft_head_gb300 import binding
from speculative_decoding_draft_head_gb300.synth import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


def test_bounded_waits_give_up_and_report():
    t0 = time.perf_counter()
    assert binding.selftest_bounded_wait(2000) == 3
    assert time.perf_counter() - t0 >= 2e-3  # both waits ran to their limit (about 2 ms each)
    # the context is still usable: a draft call runs and repeats bit for bit
    w = WORKLOADS["dspark5"].scaled(B=8, V=2056)
    inp = make_inputs(w, 0, device="cuda")
    outs = []
    for _ in range(2):
        d = binding.draft_sample(inp["base"], inp["e_in"], inp["w_out"], inp["anchor"], inp["temperature"],
                                 inp["request_id"], 0)
        torch.cuda.synchronize()
        outs.append(d["tokens"].cpu().numpy())
    assert np.array_equal(outs[0], outs[1]) and outs[0].min() >= 0


def test_selftest_rejects_bad_limits():
    with pytest.raises(binding.DSparkError):
        binding.selftest_bounded_wait(0)
    with pytest.raises(binding.DSparkError):
        binding.selftest_bounded_wait(2_000_000)

