"""Masked vocabulary entries against the oracle.

Serving engines mask tokens (vocabulary padding, banned tokens) by giving them
a very low logit.  The draft adds the base logits on the tensor cores and both
softmaxes keep a running reference that may lag the maximum, so a row whose
first values are masked exercises the renormalisation paths of the draft, the
target-row statistics and the final draw.  The masked value is large and
finite: -3e4, far below every unmasked logit (an IEEE -inf base logit is not
supported: the tensor-core base add multiplies it by zero).
"""
import numpy as np
import pytest

import oracle
from speculative_decoding_draft_head_gb300 import binding
from speculative_decoding_draft_head_gb300.synth import WORKLOADS, make_inputs

from parity import Tally, compare_draft, compare_schedule, compare_verify, gpu_round, host_inputs, oracle_round

pytestmark = pytest.mark.gpu

MASK = -3.0e4

CASES = {
    # bf16 tensor-core path: 3 row tiles, ragged vocabulary tail
    "bf16": WORKLOADS["highconc"].scaled(B=150, G=4, V=4104, r=64),
    # fp32 CUDA-core path, greedy and sampled requests
    "f32": WORKLOADS["largev"].scaled(B=24, G=5, V=2056, r=32, dtype="f32"),
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    binding.load()
    oracle.build()


def _mask(inp, V, seed):
    rng = np.random.default_rng(seed)
    head = 200 + 8 * int(rng.integers(0, 40))            # a masked vocabulary head ...
    tail = 8 * int(rng.integers(1, 20))                  # ... and a padded tail
    for k in ("base", "target"):
        inp[k][..., :head] = MASK
        inp[k][..., V - tail:] = MASK
    # tokens the target alone bans: the draft may still propose them (p = 0)
    banned = rng.choice(np.arange(head, V - tail), size=64, replace=False)
    inp["target"][..., banned] = MASK
    return head, tail


@pytest.mark.parametrize("case", list(CASES))
@pytest.mark.parametrize("seed", [0, 1])
def test_masked_tokens_match_oracle_and_are_never_emitted(case, seed):
    w = CASES[case]
    inp = make_inputs(w, seed, device="cuda")
    head, tail = _mask(inp, w.V, seed)
    g = gpu_round(inp, w, seed)
    h = host_inputs(inp)
    o = oracle_round(h, w, seed)
    temps = h["temperature"].numpy()
    t = Tally()
    td, diverged = compare_draft(g["draft"], o["draft"], temps, o["reqs"])
    t.add(td)
    skip = diverged.copy()
    if w.scheduler:
        t.add(compare_schedule(g["sched"], o["sched"]))
        skip |= g["sched"]["verify_len"].numpy() != o["sched"]["verify_len"]
    t.add(compare_verify(g["verify"], o["verify"], temps, o["reqs"], skip))
    t.check()
    assert t.exempt <= t.allowed_exempt()
    # a masked token has probability 2^-40000 or less: never drafted, never emitted
    tok = g["draft"]["tokens"].numpy()
    out = g["verify"]["out_tokens"].numpy()
    n = g["verify"]["num_out"].numpy()
    for b in range(w.B):
        for x in list(tok[b]) + list(out[b, :n[b]]):
            assert head <= x < w.V - tail
    assert np.all(np.isfinite(g["draft"]["lse"].numpy()))
